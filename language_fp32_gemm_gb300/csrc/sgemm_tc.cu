// Tensor-core SGEMM for sm_103a: C = alpha * A * B + beta * C on the
// fifth-generation tensor cores, with operands split into tf32 pairs.
//
// What is computed (the accumulator-tile kernel of the "@cluster" attribute
// page, `matmul` listing; "Show HN: Phobos", "Matrix Multiplication"): one CTA
// owns a 128 x BN tile of C, loops over K in blocks of 32, accumulates
// acc += A[tile rows, k block] * B[k block, tile cols], and stores
// alpha * acc + beta * C_old once at the end.
//
// How it maps onto GB300:
//  - Operand K-panels arrive by TMA into an S-stage shared-memory ring with
//    128-byte swizzling, gated by full/empty mbarriers (the pages' "@pipeline"
//    ping-pong buffering, generalised to S stages).
//  - One thread issues tcgen05.mma (kind::tf32, M = 128, N = BN, K = 8) into a
//    tensor-memory (TMEM) accumulator; a commit to the stage's empty barrier
//    releases the slot to the producer.
//  - Split TF32 (passes = 3): a = a_big + a_small with both parts rounded to
//    tf32 by the pre-pass, and acc += a_small*b_big + a_big*b_small +
//    a_big*b_big per K = 8 slice; the dropped a_small*b_small term is below
//    2^-22 |a||b|.  passes = 1 issues a_big*b_big only.
//  - Promotion: the tensor core's fp32 accumulation rounds towards zero, which
//    biases long sums (measured on GB300: at K = 8192 the split-TF32 error
//    reached 3.7e-6 of sum|a||b| for random signs, and a -8.6e-5 mean bias for
//    positive data).  So TMEM only holds a partial sum over `promote_blocks`
//    K blocks (1 to 8 for split TF32, shorter when K is short).  Two TMEM buffers alternate: while
//    the MMAs fill one, eight epilogue warps read the other with tcgen05.ld and
//    add it into fp32 registers with round-to-nearest adds.  This is the
//    remedy of Ootomo & Yokota (2022) for tensor-core accumulation, done with
//    TMEM double buffering.  The tile's final sum therefore lives in registers
//    (128 lanes x BN columns spread over 256 threads), the same place the
//    pages' codegen puts a CTA-wide accumulator tile.
//  - Epilogue: fmaf(alpha, sum, beta * c_old).  Aligned C takes 16-byte
//    row-segment stores; any other ldc or edge goes through a per-warp 32 x 32
//    shared-memory transpose so every access is a coalesced row segment.  The
//    old C values of a block are loaded before any store.
//
//  - CTA pairs (PAIR = true): a thread-block cluster of two CTAs on the two
//    SMs of one TPC computes a 256 x BN tile with tcgen05.mma.cta_group::2
//    (the CTA-pair mode of the "Clusters et DSMEM" chapter, section 3.4: the
//    tile grows from 128 x 128 to 256 x 128, here 256 x 256).  Each CTA TMA-loads
//    its own 128 rows of A and its own BN/2 rows of B; the leader CTA's
//    barrier counts both CTAs' bytes, the leader alone issues the MMAs, and
//    each SM reads its B half once for both tensor cores, which halves the
//    per-SM operand traffic of the single-CTA tile.  Commits are multicast to
//    both CTAs; the peer's epilogue warps arrive on the leader's barriers
//    through distributed shared memory.
//  - Multicast clusters (MC = true, an opt-in plan): a cluster of four CTAs
//    holds two pairs that compute horizontally adjacent tiles, i.e. one
//    super-tile of 256 x 512 (the "@cluster" page's super-tile as a
//    thread-block cluster; "Clusters et DSMEM", section 3.5, TMA multicast).
//    Both pairs need the same A rows: each pair TMA-loads half of them and
//    multicasts them into the rings of both pairs, so A crosses from L2 once
//    per two tiles.  A ring slot is free once both pairs' MMAs have read it:
//    each leader's commit arrives on the empty barriers of all four CTAs.
//
// The kernel is persistent: one CTA (or CTA pair) per SM (pair) loops over the
// output tiles with a static stride.  Ring slots, phases and TMEM buffers run
// on across tiles, so the next tile's loads and MMAs start while the epilogue
// warps still store the previous tile from registers.
//
// Warp roles (320 threads): warp 0 = TMA producer, warp 1 = TMEM allocator and
// MMA issuer, warps 2..9 = accumulator/epilogue warps; with A split inside the
// kernel (384 threads), the producer TMA-loads the caller's raw fp32 A (zero
// fill outside the matrix) and warps 10 and 11 split each landed tile in place
// into tf32 big/small before the MMA issuer may use it.  Epilogue warp w reads
// TMEM lanes 32*(w%4) .. +31 (the hardware's lane-quarter rule) and columns
// [h*BN/2, (h+1)*BN/2) with h = (w-2)/4.
#include "internal.h"
#include "ptx.cuh"

namespace phobos {

namespace {

constexpr int kBM = 128;  // A rows (and output rows) per CTA
constexpr int kBK = 32;   // fp32 elements per row of one stage = 128 bytes = swizzle span
constexpr int kEpiWarps = 8;
constexpr int kThreads = 64 + 32 * kEpiWarps;
constexpr int kCvtWarps = 2;  // warps 10, 11: split A in shared memory (in-kernel A split)
constexpr int threads_for(bool asplit) { return kThreads + (asplit ? 32 * kCvtWarps : 0); }
constexpr int kSmemLimit = 227 * 1024;
constexpr uint64_t kAbortGraceNs = 200000;  // let copies in flight land before exit
// With A split inside the kernel, the producer asks L2 for the caller's raw A
// this many k blocks ahead of its loads. Each raw A tile is read once, from
// HBM, and its stage then waits for the split and the pair's relay, so the
// load itself has little slack. Measured on GB300: 2 to 8 blocks ahead give
// the same gain (about 10 % at 65536x256x4096). Prefetching the pre-split
// operands of the other path, which are re-read from L2, made it slower.
constexpr int kRawAPrefetchAhead = 2;

template <int BN, int PASSES, bool PAIR>
struct TcShape {
  static constexpr int kOps = PASSES == 3 ? 2 : 1;   // big (+ small) per operand
  static constexpr int kBRows = PAIR ? BN / 2 : BN;  // B rows this CTA loads
  static constexpr int kATile = kBM * kBK * 4;        // 16 KiB
  static constexpr int kBTile = kBRows * kBK * 4;
  static constexpr int kStageBytes = kOps * (kATile + kBTile);
  static constexpr int kTmemCols = 2 * BN;            // two accumulator buffers
  // alignment slack + barriers + the accumulator warps' 32 x 32 transpose buffers
  static constexpr int kAux = 1024 + 256 + kEpiWarps * 32 * 32 * 4;
  static constexpr int max_stages() { return (kSmemLimit - kAux) / kStageBytes; }
  static constexpr int smem_bytes(int stages) { return stages * kStageBytes + kAux; }
};

__device__ __forceinline__ void raster(int t, int tiles_m, int tiles_n, int group_m, int &tm,
                                       int &tn) {
  // Output tiles are walked super-tile by super-tile: group_m tile rows at a
  // time, column by column inside the group, so that the CTAs resident at one
  // time share A row panels and B column panels in L2.
  const int per_group = group_m * tiles_n;
  const int g = t / per_group;
  const int first = g * group_m;
  const int rows = min(group_m, tiles_m - first);
  const int r = t - g * per_group;
  tm = first + r % rows;
  tn = r / rows;
}

// One unit of work of a persistent CTA (pair): a whole tile (piece = -1), or
// one K piece of a tail tile: piece 0 starts at k = 0 and owns the tile (it
// adds the other pieces and stores C), piece 1 is any later piece (its sum goes
// to partials slot `worker`).
struct Unit {
  int tile, k_lo, k_hi, piece;
};

// The i-th unit of worker w out of `units`: whole tiles w, w + units, ... below
// full_tiles, then the pieces of its share of the tail (the host deals the
// tail's K blocks to tail_units workers): at most two, since a share is shorter
// than a tile (the end of one tail tile, then the start of the next).  A later
// piece is always the first piece of its worker, so it never waits on
// anything; only piece 0 waits, for later pieces, which every worker reaches
// right after its whole tiles.  Every role of the CTA walks the same sequence.
__device__ __forceinline__ bool unit_of(const TcArgs &p, int w, int units, int i, Unit &u) {
  const int total = p.tiles_m * p.tiles_n;
  if (p.tail_units <= 0) {
    const int t = w + i * units;
    if (t >= total) return false;
    u = Unit{t, 0, p.k_blocks, -1};
    return true;
  }
  const int n_whole = p.full_tiles > w ? (p.full_tiles - w + units - 1) / units : 0;
  if (i < n_whole) {
    u = Unit{w + i * units, 0, p.k_blocks, -1};
    return true;
  }
  const int j = i - n_whole;
  if (w >= p.tail_units || j > 1) return false;
  const int st = p.tail_tile[w], sk = p.tail_k[w];
  const int et = p.tail_tile[w + 1], ek = p.tail_k[w + 1];
  if (st > et || (st == et && sk >= ek)) return false;  // an empty share
  if (j == 0) {
    u.tile = p.full_tiles + st;
    u.k_lo = sk;
    u.k_hi = et > st ? p.k_blocks : ek;
    u.piece = sk == 0 ? 0 : 1;
    return true;
  }
  if (et != st + 1 || ek == 0) return false;  // the share ends inside (or at the end of) its first tile
  u = Unit{p.full_tiles + st + 1, 0, ek, 0};
  return true;
}

// Walks the same (unit, k block) sequence as the loads of the caller's raw A,
// ahead of them, and prefetches each k block's A box into L2.
template <bool PAIR>
struct RawAPrefetch {
  static constexpr int kTileM = PAIR ? 2 * kBM : kBM;
  int i = 0, kb = 0, m0 = 0;
  bool valid = false;
  Unit u;

  __device__ __forceinline__ void start(const TcArgs &p, int w, int units, uint32_t rank) {
    valid = unit_of(p, w, units, 0, u);
    if (valid) enter(p, rank);
  }
  __device__ __forceinline__ void enter(const TcArgs &p, uint32_t rank) {
    int tm, tn;
    raster(u.tile, p.tiles_m, p.tiles_n, p.group_m, tm, tn);
    m0 = tm * kTileM + static_cast<int>(rank) * kBM;
    kb = u.k_lo;
  }
  // Prefetch the current k block's box (when it starts inside A), then step.
  __device__ __forceinline__ void step(const TcArgs &p, int w, int units, uint32_t rank) {
    if (!valid) return;
    if (m0 < p.M) tma_prefetch_2d(&p.tmap_ab, (p.k_block0 + kb) * kBK, m0);
    if (++kb >= u.k_hi) {
      valid = unit_of(p, w, units, ++i, u);
      if (valid) enter(p, rank);
    }
  }
};

// ------------------------------------------------- in-kernel panel split
// The order in which the splitter warps take the items of the split (see
// TcArgs::split_inline): by the wave of the persistent walk that first needs a
// panel, then by K chunk, then by panel and slice.  Wave v holds tiles
// [v * units, (v + 1) * units) of the raster walk; the panels first needed in
// wave v are those not needed by an earlier tile.
struct SplitOrder {
  int units, total, group_m, per_group, rows0, tiles_m, tiles_n, kc_n, waves;
  bool with_b;
  long long items;

  __device__ __forceinline__ void init(const TcArgs &p, int units_) {
    units = units_;
    total = p.tiles_m * p.tiles_n;
    group_m = p.group_m;
    per_group = p.group_m * p.tiles_n;
    rows0 = min(p.group_m, p.tiles_m);
    tiles_m = p.tiles_m;
    tiles_n = p.tiles_n;
    kc_n = (p.k_blocks + kSplitChunkBlocks - 1) / kSplitChunkBlocks;
    waves = (total + units - 1) / units;
    with_b = p.split_b != 0;
    items = static_cast<long long>(kc_n) * 8 * (tiles_m + (with_b ? tiles_n : 0));
  }
  // A panels (tile rows) first needed by a tile of index < t: in group g the
  // walk visits rows first .. first + rows - 1 in its first column.
  __device__ __forceinline__ int a_count(long long t) const {
    if (t >= total) return tiles_m;
    const int g = static_cast<int>(t / per_group);
    const int r = static_cast<int>(t - static_cast<long long>(g) * per_group);
    const int first = g * group_m;
    return first + min(r, min(group_m, tiles_m - first));
  }
  // B panels (tile columns) first needed by a tile of index < t: column tn
  // first appears at tile tn * rows0 of the first group.
  __device__ __forceinline__ int b_count(long long t) const {
    if (!with_b) return 0;
    if (t >= total) return tiles_n;
    return static_cast<int>(min(static_cast<long long>(tiles_n), (t + rows0 - 1) / rows0));
  }
  __device__ __forceinline__ long long base(int v) const {
    const long long t = static_cast<long long>(v) * units;
    return static_cast<long long>(kc_n) * 8 * (a_count(t) + b_count(t));
  }
  // Item i -> wave, operand (0 = A, 1 = B), panel, K chunk and 32-wide slice.
  __device__ __forceinline__ void item(long long i, int &wave, int &is_b, int &panel, int &kc,
                                       int &slice) const {
    int lo = 0, hi = waves;  // base(lo) <= i < base(hi) = items
    while (hi - lo > 1) {
      const int mid = (lo + hi) >> 1;
      if (base(mid) <= i) lo = mid;
      else hi = mid;
    }
    wave = lo;
    const long long t0 = static_cast<long long>(lo) * units, t1 = t0 + units;
    const int a0 = a_count(t0), a1 = a_count(t1), b0 = b_count(t0), b1 = b_count(t1);
    const int per_kc = 8 * ((a1 - a0) + (b1 - b0));
    const long long o = i - base(lo);
    kc = static_cast<int>(o / per_kc);
    const int rem = static_cast<int>(o - static_cast<long long>(kc) * per_kc);
    const int pi = rem >> 3;
    slice = rem & 7;
    if (pi < a1 - a0) {
      is_b = 0;
      panel = a0 + pi;
    } else {
      is_b = 1;
      panel = b0 + (pi - (a1 - a0));
    }
  }
};

// x -> tf32 pair: big = rna_tf32(x), small = rna_tf32(x - big) (exact difference).
__device__ __forceinline__ void split4(const float4 &x, float4 &big, float4 &small) {
  big.x = tf32_rna_bits(x.x); small.x = tf32_rna_bits(x.x - big.x);
  big.y = tf32_rna_bits(x.y); small.y = tf32_rna_bits(x.y - big.y);
  big.z = tf32_rna_bits(x.z); small.z = tf32_rna_bits(x.z - big.z);
  big.w = tf32_rna_bits(x.w); small.w = tf32_rna_bits(x.w - big.w);
}

// Up to four elements x[k .. k+3] of a row of the caller's matrix (zeros at
// and beyond `k_end`), as one 16-byte load when `vec` allows.
__device__ __forceinline__ float4 load_row4(const float *row, int k, int k_end, bool vec) {
  float4 x = make_float4(0.f, 0.f, 0.f, 0.f);
  if (vec && k + 3 < k_end) return __ldg(reinterpret_cast<const float4 *>(row + k));
  if (k < k_end) x.x = __ldg(row + k);
  if (k + 1 < k_end) x.y = __ldg(row + k + 1);
  if (k + 2 < k_end) x.z = __ldg(row + k + 2);
  if (k + 3 < k_end) x.w = __ldg(row + k + 3);
  return x;
}

// Loads in flight per lane of a splitter warp: the items are latency-bound
// (two warps per SM), so each lane issues this many 16-byte loads before it
// uses the first.  32 made the items slower on GB300 (the 128 registers of
// data no longer fit beside the rest of the kernel's 168).
constexpr int kSplitLoads = 16;

// One A item: rows r0 .. r0+31 over K [k0, k1) into the K-major workspace
// rows (zeros past M and K).  Element e of the item is (row e / G, float4
// group e % G), G = the item's float4 groups per row: each load and store
// instruction of the warp covers whole 128-byte row segments.
template <int PASSES>
__device__ __forceinline__ void split_a_item(const TcArgs &p, int r0, int k0, int k1, int lane) {
  constexpr int kGroups = kSplitChunkBlocks * kBK / 4;  // float4 groups per row of a whole item
  const int groups = (k1 - k0) >> 2;                    // ... of this item (K tail: fewer)
  constexpr int kBatches = 32 * kGroups / 32 / kSplitLoads;
  static_assert(kBatches >= 1 && 32 * kGroups == 32 * kBatches * kSplitLoads, "whole batches");
#pragma unroll 1
  for (int b = 0; b < kBatches; ++b) {
    float4 x[kSplitLoads];
#pragma unroll
    for (int j = 0; j < kSplitLoads; ++j) {
      const int e = (b * kSplitLoads + j) * 32 + lane;
      const int row = r0 + e / kGroups, c = e % kGroups;
      x[j] = make_float4(0.f, 0.f, 0.f, 0.f);
      if (c < groups && row < p.M)
        x[j] = load_row4(p.A_raw + static_cast<int64_t>(row) * p.lda, k0 + 4 * c, p.K, p.vec_a);
    }
#pragma unroll
    for (int j = 0; j < kSplitLoads; ++j) {
      const int e = (b * kSplitLoads + j) * 32 + lane;
      const int row = r0 + e / kGroups, c = e % kGroups;
      if (c < groups) {
        float4 big, small;
        split4(x[j], big, small);
        const int64_t o = static_cast<int64_t>(row) * p.kp + k0 + 4 * c;
        *reinterpret_cast<float4 *>(p.a_big + o) = big;
        if (PASSES == 3) *reinterpret_cast<float4 *>(p.a_small + o) = small;
      }
    }
  }
}

// One B item: columns n0 .. n0+31 of B over K [k0, k1), written transposed
// (row n of the workspace holds column n of B).  Lane (c, q) = (lane % 8,
// lane / 8) loads rows k = 8q .. 8q+7 of a 32-deep K block at columns
// n0 + 4c .. +3 (each load instruction covers four 128-byte row segments),
// so it holds an 8 x 4 block and writes each of its four columns as 32
// contiguous bytes of K; the lanes of one q together cover 128 bytes of a
// workspace row.  kSplitLoads / 8 K blocks are in flight at once.
template <int PASSES>
__device__ __forceinline__ void split_b_item(const TcArgs &p, int n0, int k0, int k1, int lane) {
  const int c = lane & 7, q = lane >> 3;
  const int n = n0 + 4 * c;
  const bool vec = p.vec_b && n + 3 < p.N;
  constexpr int kBlocks = kSplitLoads / 8;  // 32-deep K blocks per batch
#pragma unroll 1
  for (int kr = k0; kr < k1; kr += 32 * kBlocks) {
    float4 x[kSplitLoads];
#pragma unroll
    for (int j = 0; j < kSplitLoads; ++j) {
      const int k = kr + 32 * (j >> 3) + 8 * q + (j & 7);
      x[j] = make_float4(0.f, 0.f, 0.f, 0.f);
      if (k < k1 && k < p.K) {
        const float *src = p.B_raw + static_cast<int64_t>(k) * p.ldb;
        if (vec) {
          x[j] = __ldg(reinterpret_cast<const float4 *>(src + n));
        } else {
          if (n < p.N) x[j].x = __ldg(src + n);
          if (n + 1 < p.N) x[j].y = __ldg(src + n + 1);
          if (n + 2 < p.N) x[j].z = __ldg(src + n + 2);
          if (n + 3 < p.N) x[j].w = __ldg(src + n + 3);
        }
      }
    }
#pragma unroll
    for (int h = 0; h < kBlocks; ++h) {
      const int kb = kr + 32 * h + 8 * q;
      if (kr + 32 * h >= k1) break;  // k1 - k0 is a multiple of 32
#pragma unroll
      for (int t = 0; t < 4; ++t) {
        // column n + t of the 8 x 4 block: K kb .. kb+7
        auto col = [&](int i) {
          const float4 &v = x[8 * h + i];
          return t == 0 ? v.x : t == 1 ? v.y : t == 2 ? v.z : v.w;
        };
        float4 big0, small0, big1, small1;
        split4(make_float4(col(0), col(1), col(2), col(3)), big0, small0);
        split4(make_float4(col(4), col(5), col(6), col(7)), big1, small1);
        const int64_t o = static_cast<int64_t>(n + t) * p.kp + kb;
        *reinterpret_cast<float4 *>(p.b_big + o) = big0;
        *reinterpret_cast<float4 *>(p.b_big + o + 4) = big1;
        if (PASSES == 3) {
          *reinterpret_cast<float4 *>(p.b_small + o) = small0;
          *reinterpret_cast<float4 *>(p.b_small + o + 4) = small1;
        }
      }
    }
  }
}

// Splits item i and publishes its flag (every lane of the warp takes part).
template <int PASSES>
__device__ __forceinline__ void split_item(const TcArgs &p, const SplitOrder &ord, long long i,
                                           int lane) {
  int wave, is_b, panel, kc, slice;
  ord.item(i, wave, is_b, panel, kc, slice);
  const int kb0 = kc * kSplitChunkBlocks;
  const int kb1 = min(p.k_blocks, kb0 + kSplitChunkBlocks);
  const int k0 = (p.k_block0 + kb0) * kBK, k1 = (p.k_block0 + kb1) * kBK;
  if (is_b)
    split_b_item<PASSES>(p, panel * 256 + slice * 32, k0, k1, lane);
  else
    split_a_item<PASSES>(p, panel * 256 + slice * 32, k0, k1, lane);
  // Every lane's stores visible (to the TMA's async proxy too), then the flag.
  __threadfence();
  fence_proxy_async_global();
  __syncwarp();
  // (failure-detection test: the first item's flag is never published, so a
  // producer's bounded wait for it expires and the kernel aborts)
  if (lane == 0 && !(p.withhold_first_load == 2 && i == 0)) {
    const long long f =
        (static_cast<long long>(is_b ? ord.tiles_m + panel : panel) * ord.kc_n + kc) * 8 + slice;
    st_release_gpu(p.split_flags + f, p.epoch);
    red_release_gpu_add(p.split_done + (p.epoch - 1), 1u);
  }
}

// Splitter warp: claims items in order, splits each, publishes its flag.
// Never waits on another role, so the producers that wait on its flags always
// make progress; stops early only when the CTA aborts.
template <int PASSES>
__device__ void run_splitter(const TcArgs &p, int units, int lane, volatile int *abort_flag) {
  SplitOrder ord;
  ord.init(p, units);
  unsigned *next = p.split_next + (p.epoch - 1);
  long long i = 0;
  if (lane == 0) i = atomicAdd(next, 1u);
  i = __shfl_sync(0xffffffffu, i, 0);
  while (i < ord.items && !*abort_flag) {
    // claim the following item now, so that the atomic's round trip overlaps
    // this item's loads
    unsigned claimed = 0;
    if (lane == 0) claimed = atomicAdd(next, 1u);
    split_item<PASSES>(p, ord, i, lane);
    i = __shfl_sync(0xffffffffu, static_cast<long long>(claimed), 0);
  }
}

// Producer side: wait until the four A slices and four B slices that this
// CTA loads for K chunk kc of tile (tm, tn) are split.  Bounded like every
// wait of the kernel.
__device__ __forceinline__ bool wait_split_chunk(const TcArgs &p, int tm, int tn, int kc,
                                                 uint32_t rank, volatile int *abort_flag,
                                                 bool &all_split) {
  const int kc_n = (p.k_blocks + kSplitChunkBlocks - 1) / kSplitChunkBlocks;
  // every item of this launch (far below 2^32 for any problem that fits the
  // device: each is 32 x 256 elements of A or B)
  const unsigned items =
      static_cast<unsigned>(kc_n) * 8u * static_cast<unsigned>(p.tiles_m + (p.split_b ? p.tiles_n : 0));
  const unsigned *fa = p.split_flags + (static_cast<long long>(tm) * kc_n + kc) * 8 + 4 * rank;
  const unsigned *fb =
      p.split_flags + (static_cast<long long>(p.tiles_m + tn) * kc_n + kc) * 8 + 4 * rank;
  const unsigned e = p.epoch;
  auto ready = [&]() {
    const unsigned done = ld_relaxed_gpu(p.split_done + (e - 1));
    const unsigned a0 = ld_relaxed_gpu(fa), a1 = ld_relaxed_gpu(fa + 1);
    const unsigned a2 = ld_relaxed_gpu(fa + 2), a3 = ld_relaxed_gpu(fa + 3);
    bool ok = a0 == e && a1 == e && a2 == e && a3 == e;
    if (p.split_b) {
      const unsigned b0 = ld_relaxed_gpu(fb), b1 = ld_relaxed_gpu(fb + 1);
      const unsigned b2 = ld_relaxed_gpu(fb + 2), b3 = ld_relaxed_gpu(fb + 3);
      ok = ok && b0 == e && b1 == e && b2 == e && b3 == e;
    }
    if (done == items) all_split = true;  // no later chunk needs a wait
    return ok || all_split;
  };
  if (!ready()) {
    const uint64_t t0 = globaltimer_ns();
    for (uint32_t polls = 1; !ready(); ++polls) {
      if (*abort_flag) return false;
      if (polls >= kWaitLimitPolls || globaltimer_ns() - t0 > kWaitLimitNs) {
        *abort_flag = 1;
        atomicCAS(p.err, 0, kDevTimeoutSplit);
        return false;
      }
    }
  }
  fence_acq_rel_gpu();         // the flags' (or the count's) acquire: the split
  fence_proxy_async_global();  // stores happen-before the TMA loads issued after this
  return true;
}

template <int BN, int PASSES, int STAGES, bool PAIR, bool ASPLIT, int KIND = kTcTf32,
          bool MC = false, bool INL = false, bool CLC = false>
__global__ void __launch_bounds__(threads_for(ASPLIT || INL), 1)
    sgemm_tc_kernel(const __grid_constant__ TcArgs p) {
  using S = TcShape<BN, PASSES, PAIR>;
  static_assert(KIND == kTcTf32 || (PASSES == 1 && !ASPLIT), "16-bit inputs: one pass, pre-converted");
  static_assert(!MC || (PAIR && !ASPLIT && KIND == kTcTf32), "multicast: pre-split tf32 pairs");
  static_assert(!INL || (PAIR && !ASPLIT && !MC && KIND == kTcTf32),
                "in-kernel panel split: tf32 CTA pairs without multicast");
  static_assert((4 * STAGES + 5) * 8 + 8 <= 256, "barriers, TMEM slot and abort flag fit 256 bytes");
  // K elements per 128-byte stage row: 32 fp32/tf32 or 64 fp16/bf16.
  constexpr int kBKE = KIND == kTcTf32 ? kBK : 2 * kBK;
  constexpr int kHalf = BN / 2;  // columns summed by one epilogue thread
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t tiles = (raw + 1023u) & ~1023u;  // 1024-byte aligned stage ring
  uint8_t *aux = smem_raw + (tiles - raw) + STAGES * S::kStageBytes;
  uint64_t *bars = reinterpret_cast<uint64_t *>(aux);
  // bars: [0,S) full, [S,2S) empty, 2S+{0,1} acc_full, 2S+{2,3} acc_empty, 2S+4 MMA drained,
  // then (in-kernel A split) [2S+5, 3S+5) a_full, [3S+5, 4S+5) converted
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(bars + 4 * STAGES + 5);
  volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_slot + 1);
  // Cluster Launch Control state after the abort flag (16-byte aligned): the
  // hardware's answer and its barrier, then a two-entry ring of tile indices
  // with full barriers (both CTAs) and empty barriers (the leader's).
  static_assert(!CLC || (PAIR && !ASPLIT && !MC && (4 * STAGES + 5) * 8 + 8 + 64 <= 256),
                "Cluster Launch Control: CTA pairs without multicast or the A split in shared "
                "memory, and room for its state in the barrier block");
  const uint32_t clc_resp = smem_u32(tmem_slot + 2);
  const uint32_t clc_full = clc_resp + 16u;
  const uint32_t tile_full0 = clc_resp + 24u;
  const uint32_t tile_empty0 = clc_resp + 40u;
  const uint32_t tile_ring0 = clc_resp + 56u;
  float *epi_stage = reinterpret_cast<float *>(aux + 256);  // kEpiWarps x 32 x 32 floats

  const uint32_t full0 = smem_u32(bars);
  const uint32_t empty0 = full0 + 8u * STAGES;
  const uint32_t acc_full0 = full0 + 16u * STAGES;
  const uint32_t acc_empty0 = acc_full0 + 16u;
  const uint32_t mma_drained = acc_full0 + 32u;
  const uint32_t a_full0 = mma_drained + 8u;     // this CTA's raw A tile landed
  const uint32_t conv0 = a_full0 + 8u * STAGES;  // A tile split (leader: both CTAs)

  // (instrumentation) the SM clock over this CTA's lifetime, in CTA 0 only
  const bool clock_probe = p.clock_acc != nullptr && blockIdx.x == 0 && threadIdx.x == 0;
  long long probe_cycles = 0;
  uint64_t probe_ns = 0;
  if (clock_probe) {
    probe_ns = globaltimer_ns();
    probe_cycles = clock64();
  }

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  // Cluster layout: one CTA, one CTA pair (ranks 0, 1), or with multicast two
  // pairs (ranks 0, 1 and 2, 3) that compute horizontally adjacent tiles and
  // share their A panels.
  constexpr uint32_t kCtas = MC ? 4u : PAIR ? 2u : 1u;
  const uint32_t crank = PAIR ? cluster_ctarank() : 0u;
  const uint32_t rank = MC ? (crank & 1u) : crank;  // rank inside the CTA pair
  const uint32_t pp = MC ? (crank >> 1) : 0u;       // which pair of a multicast cluster
  const uint32_t lead = MC ? (crank & ~1u) : 0u;    // cluster rank of this pair's leader
  const bool leader = rank == 0;

  // Raise the abort flag of the other CTAs of the cluster too, so all stop promptly.
  auto abort_peer = [&]() {
    const uint32_t flag = smem_u32(const_cast<int *>(abort_flag));
    if (MC) {
      for (uint32_t r = 0; r < kCtas; ++r)
        if (r != crank) st_shared_cluster_u32(mapa_shared(flag, r), 1u);
    } else if (PAIR) {
      st_shared_cluster_u32(mapa_shared(flag, rank ^ 1u), 1u);
    }
  };

  // Persistent: each CTA (pair, or pair of pairs) walks the output tiles
  // unit, unit + units, ... in raster order, so the tiles in flight at one
  // time are neighbours.  With multicast a tile of the walk is two pair tiles
  // side by side (tile columns 2 tn and 2 tn + 1); pair pp computes the second.
  constexpr int kTileM = PAIR ? 2 * kBM : kBM;
  const int unit = static_cast<int>(blockIdx.x / kCtas);
  const int units = static_cast<int>(gridDim.x / kCtas);
  auto tile_coords = [&](int t, int &tm, int &tn) {
    raster(t, p.tiles_m, p.tiles_n, p.group_m, tm, tn);
    if (MC) tn = 2 * tn + static_cast<int>(pp);
  };
  // Tail split: the partial-sum slot of worker w (one per pair of a
  // multicast cluster).
  auto slot_of = [&](int w) -> long long {
    return MC ? 2ll * w + static_cast<long long>(pp) : static_cast<long long>(w);
  };
  const int chunk = p.promote_blocks;

  // ------------------------------------------------------------ tile walk
  // Static: unit_of's stride over the persistent grid.  With Cluster Launch
  // Control the grid holds a pair per tile; a resident pair starts on its own
  // tile and its leader's producer gets every further tile from the hardware:
  // it asks (try_cancel) while it loads the current tile, then publishes the
  // answer as entry e of a two-entry ring in both CTAs.  The MMA issuer, the
  // peer's producer and every thread of the accumulator warps read the ring
  // and release the entry on the leader, one arrival each.  Entry -1 ends the
  // walk.
  constexpr bool clc = CLC;
  constexpr int kClcReaders = 2 * (1 + 32 * kEpiWarps);
  // the units the in-kernel split's item order expects to run at once
  const int walk_units = clc ? p.clc_units : units;
  bool clc_pending = false;  // (leader's producer) a request is in flight
  uint32_t clc_phase = 0;
  auto clc_request = [&]() {
    mbar_arrive_expect_tx(clc_full, 16u);
    clc_try_cancel(clc_resp, clc_full);
    clc_pending = true;
  };
  // (leader's producer) entry e >= 1: the next tile, -1 at the end, -2 when a
  // wait ran out
  auto clc_publish = [&](int e) -> int {
    int t = -1;
    if (clc_pending) {
      if (!bounded_wait(clc_full, clc_phase, abort_flag, p.err, kDevTimeoutClc)) return -2;
      clc_phase ^= 1u;
      clc_pending = false;
      const int x = clc_cancelled_ctaid_x(clc_resp);
      if (x >= 0) {
        t = x / 2;  // the first CTA of a pair has an even index
        if (t >= p.grid_units) {  // not a work item of this grid: stop, and say so
          *abort_flag = 1;
          atomicCAS(p.err, 0, kDevTimeoutClc);
          return -2;
        }
        if (p.clock_acc) atomicAdd(p.clock_acc + 2, 1ull);  // (instrumentation)
        clc_request();
      }
    }
    const uint32_t s = static_cast<uint32_t>(e - 1) & 1u;
    const uint32_t ph = (static_cast<uint32_t>(e - 1) >> 1) & 1u;
    if (!bounded_wait_cluster(tile_empty0 + 8u * s, ph ^ 1u, abort_flag, p.err, kDevTimeoutClc))
      return -2;
    st_shared_s32(tile_ring0 + 4u * s, t);
    st_shared_cluster_u32(mapa_shared(tile_ring0 + 4u * s, 1u), static_cast<uint32_t>(t));
    mbar_arrive(tile_full0 + 8u * s);
    mbar_arrive_cluster(mapa_shared(tile_full0 + 8u * s, 1u));
    return t;
  };
  // (every other reader thread) entry e >= 1, or -2 when the wait ran out
  auto clc_read = [&](int e) -> int {
    const uint32_t s = static_cast<uint32_t>(e - 1) & 1u;
    const uint32_t ph = (static_cast<uint32_t>(e - 1) >> 1) & 1u;
    if (!bounded_wait_cluster(tile_full0 + 8u * s, ph, abort_flag, p.err, kDevTimeoutClc))
      return -2;
    const int t = ld_shared_s32(tile_ring0 + 4u * s);
    if (leader)
      mbar_arrive(tile_empty0 + 8u * s);
    else
      mbar_arrive_cluster(mapa_shared(tile_empty0 + 8u * s, 0u));
    return t;
  };
  // Work item t of the grid: a whole tile, or (with clc_pieces > 1) a K
  // piece of a tile of the last partial wave (piece code 2 + q).
  auto clc_unit = [&](int t, Unit &u) {
    const int P = p.clc_pieces;
    if (P > 1 && t >= p.full_tiles) {
      const int r = t - p.full_tiles, j = r / P, qq = r - j * P;
      u = Unit{p.full_tiles + j, qq * p.k_blocks / P, (qq + 1) * p.k_blocks / P, 2 + qq};
    } else {
      u = Unit{t, 0, p.k_blocks, -1};
    }
  };
  // The i-th unit of this thread's walk; false at its end, or when a wait ran
  // out (the abort flag is then up).
  auto walk = [&](int i, Unit &u, bool publisher) -> bool {
    if constexpr (!CLC) return unit_of(p, unit, units, i, u);
    if (i == 0) {
      clc_unit(unit, u);
      return true;
    }
    const int t = publisher ? clc_publish(i) : clc_read(i);
    if (t == -2) abort_peer();
    if (t < 0) return false;
    clc_unit(t, u);
    return true;
  };

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      // multicast: every empty barrier takes both pairs' MMA commits
      mbar_init(full0 + 8u * s, 1);
      mbar_init(empty0 + 8u * s, MC ? 2 : 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(acc_full0 + 8u * b, 1);
      mbar_init(acc_empty0 + 8u * b, (PAIR ? 2 : 1) * kEpiWarps);
    }
    mbar_init(mma_drained, 1);
    if (clc) {
      mbar_init(clc_full, 1);
      for (int s = 0; s < 2; ++s) {
        mbar_init(tile_full0 + 8u * s, 1);
        mbar_init(tile_empty0 + 8u * s, kClcReaders);
      }
    }
    if (ASPLIT) {
      for (int s = 0; s < STAGES; ++s) {
        mbar_init(a_full0 + 8u * s, 1);
        // this CTA's converter warps, plus the peer's relay on the leader
        mbar_init(conv0 + 8u * s, kCvtWarps + (PAIR && leader ? 1 : 0));
      }
    }
    *abort_flag = 0;
    fence_barrier_init();
  }
  if (warp == 0 && lane == 0) {
    prefetch_tmap(&p.tmap_ab);
    prefetch_tmap(&p.tmap_bb);
    if (PASSES == 3) {
      prefetch_tmap(&p.tmap_as);
      prefetch_tmap(&p.tmap_bs);
    }
  }
  if (warp == 1) {
    if (PAIR) {
      tmem_alloc_pair(smem_u32(tmem_slot), S::kTmemCols);
      tmem_relinquish_pair();
    } else {
      tmem_alloc(smem_u32(tmem_slot), S::kTmemCols);
      tmem_relinquish();
    }
  }
  tc_fence_before();
  __syncwarp();
  if (PAIR)
    cluster_sync();  // the peer's barriers are initialised before anyone signals them
  else
    __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;

  if (INL && warp >= 2 + kEpiWarps) {
    // ------------------------------- panel splitters (in-kernel panel split)
    // Split the caller's A and B into the workspace, item by item, ahead of
    // every CTA's producer (see TcArgs::split_inline).
    run_splitter<PASSES>(p, walk_units, lane, abort_flag);
  } else if (ASPLIT && warp >= 2 + kEpiWarps) {
    // --------------------------------------- A-split warps (in-kernel split)
    // Each of the two warps converts half of every landed raw A tile in place:
    // big = rna_tf32(x) over x, small = rna_tf32(x - big) into the second A slot
    // at the same (swizzled) offset, then tells the MMA issuer (of the pair's
    // leader) that its half is ready.
    const int cw = warp - 2 - kEpiWarps;
    constexpr int kPerWarp = S::kATile / 16 / kCvtWarps;  // float4s per warp and stage
    int g = 0;
    bool ok = true;
    Unit u;
    for (int i = 0; ok && unit_of(p, unit, units, i, u); ++i) {
      for (int kb = u.k_lo; kb < u.k_hi; ++kb, ++g) {
        const int s = g % STAGES;
        const uint32_t ph = (g / STAGES) & 1u;
        if (p.withhold_first_load == 1 && g == 0) continue;  // failure-detection test
        if (!bounded_wait(a_full0 + 8u * s, ph, abort_flag, p.err, kDevTimeoutProducer)) {
          abort_peer();
          ok = false;
          break;
        }
        float4 *big = reinterpret_cast<float4 *>(smem_raw + (tiles - raw) + s * S::kStageBytes) +
                      cw * kPerWarp;
        float4 *small = big + S::kATile / 16;
        // Batches of 8 vectors: all loads first, so they overlap (the stores
        // of one vector could otherwise hold back the next vector's load).
        constexpr int kBatch = 8;
        static_assert((kPerWarp / 32) % kBatch == 0, "whole batches per warp");
#pragma unroll 1
        for (int j0 = 0; j0 < kPerWarp / 32; j0 += kBatch) {
          float4 x[kBatch];
#pragma unroll
          for (int j = 0; j < kBatch; ++j) x[j] = big[(j0 + j) * 32 + lane];
#pragma unroll
          for (int j = 0; j < kBatch; ++j) {
            float4 b, sm;
            b.x = tf32_rna_bits(x[j].x); sm.x = tf32_rna_bits(x[j].x - b.x);
            b.y = tf32_rna_bits(x[j].y); sm.y = tf32_rna_bits(x[j].y - b.y);
            b.z = tf32_rna_bits(x[j].z); sm.z = tf32_rna_bits(x[j].z - b.z);
            b.w = tf32_rna_bits(x[j].w); sm.w = tf32_rna_bits(x[j].w - b.w);
            big[(j0 + j) * 32 + lane] = b;
            if (PASSES == 3) small[(j0 + j) * 32 + lane] = sm;
          }
        }
        fence_proxy_async_shared();  // the tensor core reads these through the async proxy
        __syncwarp();
        // A CTA-scope arrive on this CTA's own barrier. In the peer, the relay
        // thread forwards it to the leader; a cluster-scope release arrive here
        // would cost the converters about 1300 cycles per stage (measured),
        // more than the stage's MMAs.
        if (lane == 0) mbar_arrive(conv0 + 8u * s);
      }
    }
  } else if (warp == 0 && ASPLIT) {
    // --------------------------- producer when A is split inside the kernel
    if (lane == 0) {
      uint32_t armed = 0, last_parity = 0;
      int g = 0;
      bool ok = true;
      Unit u;
      RawAPrefetch<PAIR> pf;
      pf.start(p, unit, units, rank);
      for (int j = 0; j < kRawAPrefetchAhead; ++j) pf.step(p, unit, units, rank);
      for (int i = 0; ok && unit_of(p, unit, units, i, u); ++i) {
        int tm, tn;
        tile_coords(u.tile, tm, tn);
        const int m0 = tm * kTileM + static_cast<int>(rank) * kBM;
        const int b_row = tn * BN + static_cast<int>(rank) * S::kBRows;
        for (int kb = u.k_lo; kb < u.k_hi; ++kb, ++g) {
          const int s = g % STAGES;
          const uint32_t ph = (g / STAGES) & 1u;
          if (p.withhold_first_load == 1 && g == 0) continue;  // failure-detection test
          if (!bounded_wait(empty0 + 8u * s, ph ^ 1u, abort_flag, p.err, kDevTimeoutProducer)) {
            abort_peer();
            ok = false;
            break;
          }
          const uint32_t full = full0 + 8u * s;
          const uint32_t af = a_full0 + 8u * s;
          const int kc = (p.k_block0 + kb) * kBKE;
          const uint32_t st = tiles + s * S::kStageBytes;
          const uint32_t bt = st + S::kOps * S::kATile;
          mbar_arrive_expect_tx(af, S::kATile);
          tma_load_2d(st, &p.tmap_ab, af, kc, m0);  // raw A, zero outside the matrix
          if (PAIR) {
            if (leader) mbar_arrive_expect_tx(full, 2 * S::kOps * S::kBTile);
            const uint32_t lead_full = mapa_shared(full, lead);
            tma_load_2d_pair(bt, &p.tmap_bb, lead_full, kc, b_row);
            if (PASSES == 3) tma_load_2d_pair(bt + S::kBTile, &p.tmap_bs, lead_full, kc, b_row);
          } else {
            mbar_arrive_expect_tx(full, S::kOps * S::kBTile);
            tma_load_2d(bt, &p.tmap_bb, full, kc, b_row);
            if (PASSES == 3) tma_load_2d(bt + S::kBTile, &p.tmap_bs, full, kc, b_row);
          }
          // after this stage's loads, so they never queue behind a prefetch
          pf.step(p, unit, units, rank);
          armed |= 1u << s;
          last_parity = (last_parity & ~(1u << s)) | (ph << s);
        }
      }
      // No bulk copy may still be writing shared memory at exit: this CTA's A
      // loads complete on its own barriers, B loads on the leader's.
      for (int s = 0; s < STAGES; ++s)
        if (armed & (1u << s)) {
          bounded_wait(a_full0 + 8u * s, (last_parity >> s) & 1u, abort_flag, p.err,
                       kDevTimeoutDrain, false);
          if (leader)
            bounded_wait(full0 + 8u * s, (last_parity >> s) & 1u, abort_flag, p.err,
                         kDevTimeoutDrain, false);
        }
      if (PAIR && *abort_flag) {
        const uint64_t t0 = globaltimer_ns();
        while (globaltimer_ns() - t0 < kAbortGraceNs) {
        }
      }
    }
  } else if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      uint32_t armed = 0, last_parity = 0;
      int g = 0;  // k blocks loaded so far by this CTA: ring slot and phase
      bool ok = true;
      bool all_split = false;  // in-kernel split: every item of the launch is done
      Unit u;
      if (clc && leader) clc_request();  // the answer is needed after this tile's loads
      for (int i = 0; ok && walk(i, u, leader); ++i) {
        int tm, tn;
        tile_coords(u.tile, tm, tn);
        const int m0 = tm * kTileM + static_cast<int>(rank) * kBM;
        const int b_row = tn * BN + static_cast<int>(rank) * S::kBRows;
        for (int kb = u.k_lo; kb < u.k_hi; ++kb, ++g) {
          const int s = g % STAGES;
          const uint32_t ph = (g / STAGES) & 1u;
          // In-kernel panel split: this CTA's rows of A and B for the K chunk
          // starting here must have been split into the workspace.
          if (INL && !all_split && (kb == u.k_lo || kb % kSplitChunkBlocks == 0) &&
              !wait_split_chunk(p, tm, tn, kb / kSplitChunkBlocks, rank, abort_flag,
                                all_split)) {
            abort_peer();
            ok = false;
            break;
          }
          // Failure-detection test: the first stage is never loaded, so the
          // MMA issuer's bounded wait on it expires and the kernel aborts.
          if (p.withhold_first_load == 1 && g == 0) continue;
          if (!bounded_wait(empty0 + 8u * s, ph ^ 1u, abort_flag, p.err, kDevTimeoutProducer)) {
            abort_peer();
            ok = false;
            break;
          }
          const uint32_t full = full0 + 8u * s;
          const int kc = (p.k_block0 + kb) * kBKE;
          const uint32_t st = tiles + s * S::kStageBytes;
          const uint32_t bt = st + S::kOps * S::kATile;
          if (MC) {
            // This CTA's 128 rows of A are the same in both pairs: each pair
            // loads half of them (64 rows) and multicasts it to the CTA of
            // the same rank in both pairs.  Every byte that lands in a pair
            // completes on its leader's full barrier, as in the pair kernel.
            // B stays per pair.
            if (leader) mbar_arrive_expect_tx(full, 2 * S::kStageBytes);
            const uint16_t mask = static_cast<uint16_t>((1u << rank) | (1u << (2u + rank)));
            const uint32_t a_dst = st + pp * (S::kATile / 2);
            const int a_row = m0 + static_cast<int>(pp) * (kBM / 2);
            const uint32_t lead_full = mapa_shared(full, lead);
            tma_load_2d_pair_multicast(a_dst, &p.tmap_ab, lead_full, kc, a_row, mask);
            if (PASSES == 3)
              tma_load_2d_pair_multicast(a_dst + S::kATile, &p.tmap_as, lead_full, kc, a_row, mask);
            tma_load_2d_pair(bt, &p.tmap_bb, lead_full, kc, b_row);
            if (PASSES == 3) tma_load_2d_pair(bt + S::kBTile, &p.tmap_bs, lead_full, kc, b_row);
          } else if (PAIR) {
            // both CTAs' bytes complete on the leader's barrier
            if (leader) mbar_arrive_expect_tx(full, 2 * S::kStageBytes);
            const uint32_t lead_full = mapa_shared(full, lead);
            tma_load_2d_pair(st, &p.tmap_ab, lead_full, kc, m0);
            if (PASSES == 3) tma_load_2d_pair(st + S::kATile, &p.tmap_as, lead_full, kc, m0);
            tma_load_2d_pair(bt, &p.tmap_bb, lead_full, kc, b_row);
            if (PASSES == 3) tma_load_2d_pair(bt + S::kBTile, &p.tmap_bs, lead_full, kc, b_row);
          } else {
            mbar_arrive_expect_tx(full, S::kStageBytes);
            tma_load_2d(st, &p.tmap_ab, full, kc, m0);
            if (PASSES == 3) tma_load_2d(st + S::kATile, &p.tmap_as, full, kc, m0);
            tma_load_2d(bt, &p.tmap_bb, full, kc, b_row);
            if (PASSES == 3) tma_load_2d(bt + S::kBTile, &p.tmap_bs, full, kc, b_row);
          }
          armed |= 1u << s;
          last_parity = (last_parity & ~(1u << s)) | (ph << s);
        }
      }
      // A cancel request still in flight (only after an abort) writes its
      // answer into shared memory: let it land before the CTA exits.
      if (CLC && clc_pending)
        bounded_wait(clc_full, clc_phase, abort_flag, p.err, kDevTimeoutDrain, false);
      // No bulk copy may still be writing shared memory at exit.  The leader's
      // full barriers count every armed stage; a pair's peer cannot observe its
      // own copies, so after an abort it gives them a bounded grace period.
      if (leader) {
        for (int s = 0; s < STAGES; ++s)
          if (armed & (1u << s))
            bounded_wait(full0 + 8u * s, (last_parity >> s) & 1u, abort_flag, p.err,
                         kDevTimeoutDrain, false);
      }
      if (PAIR && *abort_flag) {
        const uint64_t t0 = globaltimer_ns();
        while (globaltimer_ns() - t0 < kAbortGraceNs) {
        }
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issue
    if (lane == 0 && leader) {
      constexpr uint32_t idesc =
          KIND == kTcTf32 ? idesc_tf32(kTileM, BN) : idesc_f16(kTileM, BN, KIND == kTcBf16);
      int g = 0;       // k blocks consumed: ring slot and phase
      int c_glob = 0;  // partial sums produced: TMEM buffer and its phase
      bool ok = true;
      Unit u;
      for (int i = 0; ok && walk(i, u, false); ++i) {
        int kb = u.k_lo;
        const int n_chunks = (u.k_hi - u.k_lo + chunk - 1) / chunk;
        for (int c = 0; c < n_chunks && ok; ++c, ++c_glob) {
          const int b = c_glob & 1;
          const uint32_t use = static_cast<uint32_t>(c_glob >> 1);
          // the epilogue warps (of both CTAs) must have read this buffer's
          // previous partial sum
          const bool free_buf =
              PAIR ? bounded_wait_cluster(acc_empty0 + 8u * b, (use & 1u) ^ 1u, abort_flag,
                                          p.err, kDevTimeoutMma)
                   : bounded_wait(acc_empty0 + 8u * b, (use & 1u) ^ 1u, abort_flag, p.err,
                                  kDevTimeoutMma);
          if (!free_buf) {
            ok = false;
            abort_peer();
            break;
          }
          tc_fence_after();
          const uint32_t d_tmem = tmem_base + static_cast<uint32_t>(b * BN);
          const int kb_end = min(u.k_hi, kb + chunk);
          for (int first = 1; kb < kb_end; ++kb, ++g, first = 0) {
            const int s = g % STAGES;
            const uint32_t ph = (g / STAGES) & 1u;
            if (!bounded_wait(full0 + 8u * s, ph, abort_flag, p.err, kDevTimeoutMma) ||
                (ASPLIT && !(PAIR ? bounded_wait_cluster(conv0 + 8u * s, ph, abort_flag, p.err,
                                                         kDevTimeoutMma)
                                  : bounded_wait(conv0 + 8u * s, ph, abort_flag, p.err,
                                                 kDevTimeoutMma)))) {
              ok = false;
              abort_peer();
              break;
            }
            tc_fence_after();
            const uint32_t a_big = tiles + s * S::kStageBytes;
            const uint32_t a_small = a_big + S::kATile;
            const uint32_t b_big = a_big + S::kOps * S::kATile;
            const uint32_t b_small = b_big + S::kBTile;
#pragma unroll
            for (int kk = 0; kk < kBK / 8; ++kk) {
              // one MMA's K slice: 32 bytes (8 tf32, or 16 fp16/bf16)
              const uint32_t off = kk * 32u;
              const uint64_t dab = desc_kmajor_sw128(a_big + off);
              const uint64_t dbb = desc_kmajor_sw128(b_big + off);
              const uint32_t acc = (first && kk == 0) ? 0u : 1u;
              if (PASSES == 3) {
                const uint64_t das = desc_kmajor_sw128(a_small + off);
                const uint64_t dbs = desc_kmajor_sw128(b_small + off);
                if (PAIR) {
                  mma_tf32_pair(d_tmem, das, dbb, idesc, acc);
                  mma_tf32_pair(d_tmem, dab, dbs, idesc, 1u);
                  mma_tf32_pair(d_tmem, dab, dbb, idesc, 1u);
                } else {
                  mma_tf32(d_tmem, das, dbb, idesc, acc);
                  mma_tf32(d_tmem, dab, dbs, idesc, 1u);
                  mma_tf32(d_tmem, dab, dbb, idesc, 1u);
                }
              } else if (KIND == kTcTf32) {
                if (PAIR)
                  mma_tf32_pair(d_tmem, dab, dbb, idesc, acc);
                else
                  mma_tf32(d_tmem, dab, dbb, idesc, acc);
              } else {
                if (PAIR)
                  mma_f16_pair(d_tmem, dab, dbb, idesc, acc);
                else
                  mma_f16(d_tmem, dab, dbb, idesc, acc);
              }
            }
            // the slot is free once this pair's MMAs have read it; with
            // multicast both pairs' CTAs wait for both pairs' commits
            if (PAIR)
              mma_commit_pair(empty0 + 8u * s, MC ? 0xF : 0x3);
            else
              mma_commit(empty0 + 8u * s);
          }
          if (ok) {
            if (PAIR)
              mma_commit_pair(acc_full0 + 8u * b, static_cast<uint16_t>(0x3u << lead));
            else
              mma_commit(acc_full0 + 8u * b);
          }
        }
      }
      // Every MMA must be finished before TMEM is released.
      if (PAIR)
        mma_commit_pair(mma_drained, static_cast<uint16_t>(1u << lead));
      else
        mma_commit(mma_drained);
      bounded_wait(mma_drained, 0, abort_flag, p.err, kDevTimeoutDrain, false);
    } else if (ASPLIT && PAIR && lane == 0) {
      // Relay, in the peer, whose MMA warp issues nothing: once this CTA's
      // converter warps have split a stage, tell the leader's MMA issuer. The
      // release at cluster scope carries the converters' shared-memory writes
      // (ordered before it by their arrive and this thread's wait) to the
      // leader, which acquires them before its MMAs read this CTA's A.
      int g = 0;
      bool ok = true;
      Unit u;
      for (int i = 0; ok && unit_of(p, unit, units, i, u); ++i) {
        for (int kb = u.k_lo; kb < u.k_hi; ++kb, ++g) {
          const int s = g % STAGES;
          const uint32_t ph = (g / STAGES) & 1u;
          if (p.withhold_first_load == 1 && g == 0) continue;  // failure-detection test
          if (!bounded_wait(conv0 + 8u * s, ph, abort_flag, p.err, kDevTimeoutProducer)) {
            abort_peer();
            ok = false;
            break;
          }
          mbar_arrive_cluster(mapa_shared(conv0 + 8u * s, lead));
        }
      }
    }
  } else {
    // ------------------------------------------- accumulate + epilogue warps
    const int q = warp & 3;              // TMEM lane quarter this warp may read
    const int h = (warp - 2) >> 2;       // column half
    const uint32_t lane_base = static_cast<uint32_t>(q * 32) << 16;
    int c_glob = 0;
    bool ok = true;
    Unit u;
    constexpr int kRanks = PAIR ? 2 : 1;
    float *sbuf = epi_stage + (warp - 2) * 32 * 32;  // this warp's 32 x 32 block of C
    for (int i = 0; ok && walk(i, u, false); ++i) {
      int tm, tn;
      tile_coords(u.tile, tm, tn);
      // This warp owns rows row0 .. row0+31 and columns col0 .. col0+kHalf-1 of
      // the tile; lane l sums row row0 + l.
      const int tile_row = static_cast<int>(rank) * kBM + q * 32 + lane;  // 0 .. kTileM-1
      const int row0 = tm * kTileM + tile_row - lane;
      const int col0 = tn * BN + h * kHalf;
      bool writes_c = u.piece <= 0 && row0 < p.M && col0 < p.N;  // warp-uniform
      const bool vec = p.vec_c && col0 + kHalf <= p.N;            // 16-byte rows
      bool load_old = writes_c && p.beta != 0.0f;
      // Old C of columns j0 .. j0+31 into the warp's block, in the swizzled
      // layout the row-per-lane reads below use: row r, column c at
      // r*32 + (c ^ r) (4-byte copies), or 16-byte chunk ch at chunk ch ^ (r & 7).
      // Each copy instruction covers whole 128-byte row segments.
      auto fetch_old = [&](int j0) {
        if (vec) {
#pragma unroll 4
          for (int k = 0; k < 8; ++k) {
            const int r = 4 * k + (lane >> 3), ch = lane & 7;
            if (row0 + r < p.M)
              cp_async16(sbuf + r * 32 + ((ch ^ (r & 7)) << 2),
                         p.C + static_cast<int64_t>(row0 + r) * p.ldc + col0 + j0 + 4 * ch);
          }
        } else {
          const int col = col0 + j0 + lane;
          if (col < p.N) {
#pragma unroll 4
            for (int r = 0; r < 32; ++r)
              if (row0 + r < p.M)
                cp_async4(sbuf + r * 32 + (lane ^ r), p.C + static_cast<int64_t>(row0 + r) * p.ldc + col);
          }
        }
      };
      bool first_fetched = false;
      float sum[kHalf];
#pragma unroll
      for (int j = 0; j < kHalf; ++j) sum[j] = 0.f;
      const int n_chunks = (u.k_hi - u.k_lo + chunk - 1) / chunk;
      for (int c = 0; c < n_chunks; ++c, ++c_glob) {
        const int b = c_glob & 1;
        const uint32_t use = static_cast<uint32_t>(c_glob >> 1);
        if (c == n_chunks - 1 && load_old) {
          // The first block of old C does not depend on the sums: fetch it
          // while the tile's last partial sum is still being accumulated.
          fetch_old(0);
          first_fetched = true;
        }
        if (!bounded_wait(acc_full0 + 8u * b, use & 1u, abort_flag, p.err, kDevTimeoutEpilogue)) {
          ok = false;
          abort_peer();
          break;
        }
        tc_fence_after();
        const uint32_t col = tmem_base + static_cast<uint32_t>(b * BN + h * kHalf);
#pragma unroll
        for (int j = 0; j < kHalf; j += 32) {
          uint32_t r[32];
          tmem_ld32(col + lane_base + j, r);
          tmem_ld_wait(r);
#pragma unroll
          for (int u = 0; u < 32; ++u) sum[j + u] = __fadd_rn(sum[j + u], __uint_as_float(r[u]));
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) {
          if (PAIR)
            mbar_arrive_cluster(mapa_shared(acc_empty0 + 8u * b, lead));
          else
            mbar_arrive(acc_empty0 + 8u * b);
        }
      }
      if (!ok) {
        cp_async_wait_all();  // no copy may land in a buffer after the CTA exits
        break;
      }
      // Tail pieces exchange their partial sums through L2 in a warp-interleaved
      // layout: float4 v of lane l of a warp sits at (v * 32 + l), so that every
      // store and load instruction covers 512 contiguous bytes.
      if (CLC && u.piece >= 2) {
        // Cluster Launch Control tail piece q = piece - 2 of tail tile jt (see
        // TcArgs::clc_pieces): leave the partial sum in slot jt * P + q and count
        // in on the tile's counter; the last piece to arrive adds the P slots in
        // K order and stores C.  No piece waits for another, so no piece can
        // hold up a tile that the hardware has not dealt yet.
        const int P = p.clc_pieces, jt = u.tile - p.full_tiles;
        constexpr int kSlotF4 = kHalf / 4;  // float4 per lane per piece
        constexpr long long kSlotStride = static_cast<long long>(kRanks) * kEpiWarps * kSlotF4 * 32;
        float4 *const first = reinterpret_cast<float4 *>(p.partials) +
                              ((static_cast<long long>(jt) * P * kRanks + rank) * kEpiWarps +
                               (warp - 2)) * (kSlotF4 * 32) + lane;
        float4 *const mine = first + (u.piece - 2) * kSlotStride;
#pragma unroll
        for (int v = 0; v < kSlotF4; ++v)
          __stcg(mine + v * 32, make_float4(sum[4 * v], sum[4 * v + 1], sum[4 * v + 2], sum[4 * v + 3]));
        __threadfence();
        __syncwarp();
        unsigned *const counter = p.flags + (static_cast<long long>(jt) * 2 + rank) * kEpiWarps + (warp - 2);
        unsigned old = 0;
        if (lane == 0) old = atom_add_acq_rel_gpu(counter, 1u);
        old = __shfl_sync(0xffffffffu, old, 0);
        if (old + 1u != static_cast<unsigned>(P)) continue;  // a later piece finishes the tile
        (void)ld_acquire_gpu(counter);  // every lane acquires the other pieces' stores
#pragma unroll
        for (int v0 = 0; v0 < kSlotF4; v0 += 8) {
#pragma unroll 1
          for (int qq = 0; qq < P; ++qq) {
            float4 x[8];
#pragma unroll
            for (int t = 0; t < 8; ++t) x[t] = __ldcg(first + qq * kSlotStride + (v0 + t) * 32);
#pragma unroll
            for (int t = 0; t < 8; ++t) {
              const int e = 4 * (v0 + t);
              if (qq == 0) {
                sum[e] = x[t].x;
                sum[e + 1] = x[t].y;
                sum[e + 2] = x[t].z;
                sum[e + 3] = x[t].w;
              } else {
                sum[e] = __fadd_rn(sum[e], x[t].x);
                sum[e + 1] = __fadd_rn(sum[e + 1], x[t].y);
                sum[e + 2] = __fadd_rn(sum[e + 2], x[t].z);
                sum[e + 3] = __fadd_rn(sum[e + 3], x[t].w);
              }
            }
          }
        }
        __syncwarp();
        if (lane == 0) *counter = 0u;  // ready for the next launch's pieces of this tile
        writes_c = row0 < p.M && col0 < p.N;
        load_old = writes_c && p.beta != 0.0f;
      } else if (u.piece > 0) {
        // Hand the partial sum to the piece-0 owner through this worker's
        // slot, then release the flag once every accumulator thread's stores
        // are visible.
        const long long slot = slot_of(unit);
        float4 *dst = reinterpret_cast<float4 *>(p.partials) +
                      ((slot * kRanks + rank) * kEpiWarps + (warp - 2)) * (kHalf / 4) * 32 + lane;
#pragma unroll
        for (int v = 0; v < kHalf / 4; ++v)
          __stcg(dst + v * 32, make_float4(sum[4 * v], sum[4 * v + 1], sum[4 * v + 2], sum[4 * v + 3]));
        // Each warp publishes its own slice: no CTA-wide barrier, so a warp
        // that left on an abort path cannot strand the others.
        __threadfence();
        __syncwarp();
        if (lane == 0)
          st_release_gpu(p.flags + (slot * 2 + rank) * kEpiWarps + (warp - 2), p.epoch);
        continue;
      }
      if (u.piece == 0) {
        // Owner: add the later pieces of this tile in K order (deterministic).
        // They are the first pieces of the next workers, w_end excluded: the
        // host leaves no share empty, so these are consecutive.
        const int tt = u.tile - p.full_tiles;
        int w_end = unit + 1;
        while (w_end < p.tail_units && p.tail_tile[w_end] == tt) ++w_end;
        for (int w2 = unit + 1; w2 < w_end && ok; ++w2) {
          const unsigned *flag = p.flags + (slot_of(w2) * 2 + rank) * kEpiWarps + (warp - 2);
          if (ld_acquire_gpu(flag) != p.epoch) {
            const uint64_t t0 = globaltimer_ns();
            for (uint32_t polls = 1; ld_acquire_gpu(flag) != p.epoch; ++polls) {
              if ((polls & 31u) == 0 &&
                  (*abort_flag || polls >= kWaitLimitPolls || globaltimer_ns() - t0 > kWaitLimitNs)) {
                if (!*abort_flag) atomicCAS(p.err, 0, kDevTimeoutPartial);
                *abort_flag = 1;
                abort_peer();
                ok = false;
                break;
              }
            }
          }
        }
        if (!ok) {
          cp_async_wait_all();
          break;
        }
        // The pieces stream through the operand ring, which is idle now: an
        // owner piece is its worker's last unit, and its final partial sum
        // landed after every MMA of the worker had read its operands.  Each
        // lane copies and later reads only its own float4s, so no warp
        // barrier is needed; kBufs - 1 chunks are in flight while one is added
        // (registers alone held too few loads in flight: 3 to 5 us per piece).
        constexpr int kChunkF4 = 4;                     // float4 per lane per chunk
        constexpr int kSlotF4 = kHalf / 4;              // float4 per lane per piece
        constexpr int kCps = kSlotF4 / kChunkF4;        // chunks per piece
        constexpr int kRingF4PerWarp = STAGES * S::kStageBytes / 16 / kEpiWarps;
        constexpr int kBufs0 = kRingF4PerWarp / (32 * kChunkF4);
        // a power of two, at most 8
        constexpr int kBufs = kBufs0 >= 8 ? 8 : kBufs0 >= 4 ? 4 : kBufs0 >= 2 ? 2 : 0;
        static_assert(kBufs >= 2 && kSlotF4 % kChunkF4 == 0, "fix-up staging fits the ring");
        const uint32_t stage = tiles + ((warp - 2) * (kBufs * kChunkF4 * 32) + lane) * 16u;
        const float4 *part0 = reinterpret_cast<const float4 *>(p.partials) +
                              ((slot_of(unit + 1) * kRanks + rank) * kEpiWarps + (warp - 2)) *
                                  (kSlotF4 * 32) + lane;
        // the pieces' slots are consecutive (every other slot with multicast):
        // piece i of this warp at part0 + i * kSlotStride
        constexpr long long kSlotStride =
            static_cast<long long>(MC ? 2 : 1) * kRanks * kEpiWarps * kSlotF4 * 32;
        const int n_chunks = (w_end - unit - 1) * kCps;
        auto issue = [&](int c) {
          if (c < n_chunks) {
            const float4 *src = part0 + (c / kCps) * kSlotStride + (c % kCps) * (kChunkF4 * 32);
            const uint32_t dst = stage + (c % kBufs) * (kChunkF4 * 32 * 16);
#pragma unroll
            for (int q = 0; q < kChunkF4; ++q) cp_async16_u32(dst + q * 32 * 16, src + q * 32);
          }
          cp_async_commit();  // an empty group past the end keeps the count
        };
        if (n_chunks > 0) {
#pragma unroll 1
          for (int c = 0; c < kBufs - 1; ++c) issue(c);
        }
#pragma unroll 1
        for (int c0 = 0; c0 < n_chunks; c0 += kCps) {
#pragma unroll
          for (int j = 0; j < kCps; ++j) {
            const int c = c0 + j;
            issue(c + kBufs - 1);  // into the buffer of chunk c - 1, added already
            cp_async_wait_group<kBufs - 1>();  // chunk c has landed
            const uint32_t b = stage + (c % kBufs) * (kChunkF4 * 32 * 16);
#pragma unroll
            for (int q = 0; q < kChunkF4; ++q) {
              const float4 x = ld_shared_f4(b + q * 32 * 16);
              const int v = j * kChunkF4 + q;
              sum[4 * v + 0] = __fadd_rn(sum[4 * v + 0], x.x);
              sum[4 * v + 1] = __fadd_rn(sum[4 * v + 1], x.y);
              sum[4 * v + 2] = __fadd_rn(sum[4 * v + 2], x.z);
              sum[4 * v + 3] = __fadd_rn(sum[4 * v + 3], x.w);
            }
          }
        }
        cp_async_wait_all();
      }
      if (!writes_c) continue;
      // The tile's sum is in registers: TMEM already serves the next tile's
      // MMAs while this store runs.  Per 32-column block: old C lands in the
      // warp's block (asynchronous copies), each lane combines its row in
      // place, then the warp writes the block back row by row.
      const float alpha = p.alpha, beta = p.beta;
#pragma unroll
      for (int j0 = 0; j0 < kHalf; j0 += 32) {
        if (col0 + j0 >= p.N) break;  // uniform across the warp
        if (load_old) {
          if (j0 > 0 || !first_fetched) fetch_old(j0);
          cp_async_wait_all();
          __syncwarp();
        }
        if (vec) {
#pragma unroll
          for (int jj = 0; jj < 8; ++jj) {
            float4 *s4 = reinterpret_cast<float4 *>(sbuf + lane * 32 + ((jj ^ (lane & 7)) << 2));
            float4 o;
            if (load_old) {
              const float4 old = *s4;
              o.x = fmaf(alpha, sum[j0 + 4 * jj + 0], beta * old.x);
              o.y = fmaf(alpha, sum[j0 + 4 * jj + 1], beta * old.y);
              o.z = fmaf(alpha, sum[j0 + 4 * jj + 2], beta * old.z);
              o.w = fmaf(alpha, sum[j0 + 4 * jj + 3], beta * old.w);
            } else {
              o.x = alpha * sum[j0 + 4 * jj + 0];
              o.y = alpha * sum[j0 + 4 * jj + 1];
              o.z = alpha * sum[j0 + 4 * jj + 2];
              o.w = alpha * sum[j0 + 4 * jj + 3];
            }
            *s4 = o;
          }
        } else {
#pragma unroll
          for (int j = 0; j < 32; ++j) {
            float &s = sbuf[lane * 32 + (j ^ lane)];
            s = load_old ? fmaf(alpha, sum[j0 + j], beta * s) : alpha * sum[j0 + j];
          }
        }
        __syncwarp();
        if (vec) {
#pragma unroll 4
          for (int k = 0; k < 8; ++k) {
            const int r = 4 * k + (lane >> 3), ch = lane & 7;
            if (row0 + r < p.M)
              *reinterpret_cast<float4 *>(p.C + static_cast<int64_t>(row0 + r) * p.ldc + col0 + j0 +
                                          4 * ch) =
                  *reinterpret_cast<const float4 *>(sbuf + r * 32 + ((ch ^ (r & 7)) << 2));
          }
        } else {
          const int col = col0 + j0 + lane;
          if (col < p.N) {
#pragma unroll 4
            for (int r = 0; r < 32; ++r)
              if (row0 + r < p.M)
                p.C[static_cast<int64_t>(row0 + r) * p.ldc + col] = sbuf[r * 32 + (lane ^ r)];
          }
        }
        __syncwarp();
      }
    }
  }

  tc_fence_before();
  __syncwarp();
  if (PAIR)
    cluster_sync();  // the leader's MMAs read the peer's shared memory until here
  else
    __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    if (PAIR)
      tmem_dealloc_pair(tmem_base, S::kTmemCols);
    else
      tmem_dealloc(tmem_base, S::kTmemCols);
  }
  if (clock_probe) {  // every warp of the CTA has passed the barrier above
    const long long cycles = clock64() - probe_cycles;
    const uint64_t ns = globaltimer_ns() - probe_ns;
    atomicAdd(p.clock_acc, static_cast<unsigned long long>(cycles));
    atomicAdd(p.clock_acc + 1, static_cast<unsigned long long>(ns));
  }
}

// Launch configuration of one kernel instance: the persistent grid of `units`
// CTAs, CTA pairs, or (multicast) clusters of two pairs.
template <int BN, int PASSES, int STAGES, bool PAIR, bool ASPLIT, int KIND, bool MC,
          bool INL = false, bool CLC = false>
void tc_config(cudaLaunchConfig_t &cfg, cudaLaunchAttribute *attr, unsigned units,
               cudaStream_t stream) {
  using S = TcShape<BN, PASSES, PAIR>;
  const unsigned ctas = MC ? 4u : PAIR ? 2u : 1u;
  cfg = {};
  cfg.gridDim = dim3(ctas * units, 1, 1);
  cfg.blockDim = dim3(threads_for(ASPLIT || INL), 1, 1);
  cfg.dynamicSmemBytes = S::smem_bytes(STAGES);
  cfg.stream = stream;
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = ctas;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
}

template <int BN, int PASSES, int STAGES, bool PAIR, bool ASPLIT, int KIND = kTcTf32,
          bool MC = false, bool INL = false, bool CLC = false>
cudaError_t launch_one(const TcArgs &a, cudaStream_t stream) {
  using S = TcShape<BN, PASSES, PAIR>;
  static_assert(STAGES >= 2 && STAGES <= S::max_stages(), "stage ring does not fit");
  auto kern = sgemm_tc_kernel<BN, PASSES, STAGES, PAIR, ASPLIT, KIND, MC, INL, CLC>;
  const int smem = S::smem_bytes(STAGES);
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  const long long tiles = static_cast<long long>(a.tiles_m) * a.tiles_n;
  // one CTA (pair) per SM (pair), never more than there are tiles
  const long long workers = MC ? a.sm_count / 4 : PAIR ? a.sm_count / 2 : a.sm_count;
  const unsigned units = a.grid_units > 0
                             ? static_cast<unsigned>(a.grid_units)
                             : static_cast<unsigned>(tiles < workers ? tiles : workers);
  if (units == 0) return cudaErrorInvalidValue;
  if (!PAIR) {
    kern<<<units, threads_for(ASPLIT || INL), smem, stream>>>(a);
    return cudaGetLastError();
  }
  cudaLaunchConfig_t cfg;
  cudaLaunchAttribute attr[1];
  tc_config<BN, PASSES, STAGES, PAIR, ASPLIT, KIND, MC, INL, CLC>(cfg, attr, units, stream);
  return cudaLaunchKernelEx(&cfg, kern, a);
}

// Multicast clusters (two CTA pairs, four SMs) that fit on the device at once.
// The tail split makes a worker wait for others, so the persistent grid may not
// hold more clusters than can be resident together.
template <int BN, int PASSES, int STAGES>
int mc_resident_clusters(cudaStream_t stream) {
  auto kern = sgemm_tc_kernel<BN, PASSES, STAGES, true, false, kTcTf32, true>;
  const int smem = TcShape<BN, PASSES, true>::smem_bytes(STAGES);
  if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) != cudaSuccess)
    return -1;
  cudaLaunchConfig_t cfg;
  cudaLaunchAttribute attr[1];
  tc_config<BN, PASSES, STAGES, true, false, kTcTf32, true>(cfg, attr, 1, stream);
  int n = 0;
  if (cudaOccupancyMaxActiveClusters(&n, kern, &cfg) != cudaSuccess) return -1;
  return n;
}

template <int BN, int PASSES, bool PAIR>
cudaError_t launch_stages(const TcArgs &a, int stages, cudaStream_t stream, int kind) {
  constexpr int kMax = TcShape<BN, PASSES, PAIR>::max_stages();
  // Up to 6 stages: one-pass kernels (TF32, fp16, bf16) have 32 KiB stages and
  // only 512 MMA cycles per stage, so they need the deeper ring to cover a
  // load's latency; the barrier block (4 * 6 + 5 barriers) still fits its
  // 256 bytes.
  constexpr int kTop = kMax >= 6 ? 6 : kMax;
  // 16-bit inputs: one pass, pre-converted operands, the deepest ring only.
  if (kind != kTcTf32) {
    if (PASSES != 1 || a.a_inline || a.split_inline) return cudaErrorInvalidValue;
    if (stages == kTop)
      return kind == kTcF16 ? launch_one<BN, 1, kTop, PAIR, false, kTcF16>(a, stream)
                            : launch_one<BN, 1, kTop, PAIR, false, kTcBf16>(a, stream);
    if (stages == 4 && kMax >= 4)
      return kind == kTcF16 ? launch_one<BN, 1, (kMax >= 4 ? 4 : 2), PAIR, false, kTcF16>(a, stream)
                            : launch_one<BN, 1, (kMax >= 4 ? 4 : 2), PAIR, false, kTcBf16>(a, stream);
    return cudaErrorInvalidValue;
  }
  // Multicast clusters: pre-split operands, the deepest ring.
  if (a.multicast) {
    if constexpr (PAIR) {
      if (a.a_inline || a.split_inline || stages != kTop) return cudaErrorInvalidValue;
      return launch_one<BN, PASSES, kTop, true, false, kTcTf32, true>(a, stream);
    }
    return cudaErrorInvalidValue;
  }
  // Cluster Launch Control (split-TF32 CTA pairs reading A from the
  // workspace): the deepest ring, with or without the in-kernel panel split.
  if (a.clc) {
    if constexpr (PAIR && PASSES == 3) {
      if (a.a_inline || stages != kTop) return cudaErrorInvalidValue;
      return a.split_inline
                 ? launch_one<BN, 3, kTop, true, false, kTcTf32, false, true, true>(a, stream)
                 : launch_one<BN, 3, kTop, true, false, kTcTf32, false, false, true>(a, stream);
    }
    return cudaErrorInvalidValue;
  }
  // In-kernel panel split (CTA pairs): the deepest ring.
  if (a.split_inline) {
    if constexpr (PAIR) {
      if (a.a_inline || stages != kTop) return cudaErrorInvalidValue;
      return launch_one<BN, PASSES, kTop, true, false, kTcTf32, false, true>(a, stream);
    }
    return cudaErrorInvalidValue;
  }
  // In-kernel A split: always the deepest ring.
  if (a.a_inline) return launch_one<BN, PASSES, kTop, PAIR, true>(a, stream);
  if (stages >= 6 && kMax >= 6) return launch_one<BN, PASSES, (kMax >= 6 ? 6 : 2), PAIR, false>(a, stream);
  if (stages >= 5 && kMax >= 5) return launch_one<BN, PASSES, (kMax >= 5 ? 5 : 2), PAIR, false>(a, stream);
  if (stages >= 4 && kMax >= 4) return launch_one<BN, PASSES, (kMax >= 4 ? 4 : 2), PAIR, false>(a, stream);
  if (stages >= 3 && kMax >= 3) return launch_one<BN, PASSES, (kMax >= 3 ? 3 : 2), PAIR, false>(a, stream);
  if (stages >= 2) return launch_one<BN, PASSES, 2, PAIR, false>(a, stream);
  return cudaErrorInvalidValue;
}

template <bool PAIR>
int max_stages_of(int passes, int bn) {
  int m = 0;
  if (passes == 3 && bn == 256) m = TcShape<256, 3, PAIR>::max_stages();
  if (passes == 3 && bn == 128) m = TcShape<128, 3, PAIR>::max_stages();
  if (passes == 1 && bn == 256) m = TcShape<256, 1, PAIR>::max_stages();
  if (passes == 1 && bn == 128) m = TcShape<128, 1, PAIR>::max_stages();
  return m > 6 ? 6 : m;
}

}  // namespace

int tc_max_stages(int passes, int bn) { return max_stages_of<false>(passes, bn); }
int tc_pair_max_stages(int passes, int bn) { return max_stages_of<true>(passes, bn); }

int tc_multicast_clusters(int passes, int bn, cudaStream_t stream) {
  if (bn != 256) return -1;
  constexpr int k3 = TcShape<256, 3, true>::max_stages() > 6 ? 6 : TcShape<256, 3, true>::max_stages();
  constexpr int k1 = TcShape<256, 1, true>::max_stages() > 6 ? 6 : TcShape<256, 1, true>::max_stages();
  if (passes == 3) return mc_resident_clusters<256, 3, k3>(stream);
  if (passes == 1) return mc_resident_clusters<256, 1, k1>(stream);
  return -1;
}

cudaError_t launch_tc(const TcArgs &a, int passes, int bn, int stages, cudaStream_t stream,
                      int kind) {
  if (kind != kTcTf32 && kind != kTcF16 && kind != kTcBf16) return cudaErrorInvalidValue;
  if (passes == 3 && bn == 256) return launch_stages<256, 3, false>(a, stages, stream, kind);
  if (passes == 3 && bn == 128) return launch_stages<128, 3, false>(a, stages, stream, kind);
  if (passes == 1 && bn == 256) return launch_stages<256, 1, false>(a, stages, stream, kind);
  if (passes == 1 && bn == 128) return launch_stages<128, 1, false>(a, stages, stream, kind);
  return cudaErrorInvalidValue;
}

cudaError_t launch_tc_pair(const TcArgs &a, int passes, int bn, int stages, cudaStream_t stream,
                           int kind) {
  if (kind != kTcTf32 && kind != kTcF16 && kind != kTcBf16) return cudaErrorInvalidValue;
  if (passes == 3 && bn == 256) return launch_stages<256, 3, true>(a, stages, stream, kind);
  if (passes == 1 && bn == 256) return launch_stages<256, 1, true>(a, stages, stream, kind);
  return cudaErrorInvalidValue;
}

}  // namespace phobos
