// plan.cpp — host-side layout planner of libvsf.
//
// Implements the layout rule of "veScale-FSDP: Flexible and High-Performance
// FSDP at Scale (MLSys 2026)" summary page, 核心方法 › Grouped communication
// (Algorithm 1) with the atoms of 核心方法 › RaggedShard:
//   - minimise the uniform per-rank size S (Balanced Load), S a multiple of
//     g_coll (ranks start on collective units) and S >= ceil(real / m);
//   - every tensor contiguous (Contiguous Tensor Memory), padding only
//     between tensors, offsets aligned to lcm(g_coll, atom);
//   - no rank boundary inside an atom (Non-Sharded Block);
//   - tensor order: input order, atom size or element count (descending).
// The page solves placement with a monotone DP; for a fixed order, placing
// each tensor at its earliest feasible offset is exact, because the earliest
// feasible start at or after a cursor never decreases as the cursor grows.
// Feasibility is not monotone in S (one 2-atom tensor of atom 10 on 2 ranks
// fits S = 10 but not S = 11), so candidates are scanned upward.
//
// Speed: for one tensor at offset o the first boundary that cuts an atom is
// k0*S or (k0+1)*S (k0 = first boundary past o): if k0*S is on an atom
// boundary and the atom does not divide S, the next boundary is off by
// S mod atom. So one placement costs O(1) per tensor and retry.
#include <algorithm>
#include <chrono>
#include <cmath>
#include <cstring>
#include <numeric>

#include "vsf_internal.h"

namespace vsf {

namespace {
thread_local std::string g_last_error;

bool mul_ok(int64_t a, int64_t b, int64_t* out) {
  if (a < 0 || b < 0) return false;
  if (a != 0 && b > INT64_MAX / a) return false;
  *out = a * b;
  return true;
}

int64_t gcd64(int64_t a, int64_t b) { return b == 0 ? a : gcd64(b, a % b); }

int64_t round_up(int64_t x, int64_t a) {
  int64_t r = x % a;
  return r == 0 ? x : x + (a - r);
}

// Earliest feasible offset >= cursor for tensor x under per-rank size S, or
// -1 if it would end past capacity.
int64_t earliest_offset(const TensorInfo& x, int64_t S, int64_t capacity, int64_t cursor) {
  int64_t o = round_up(cursor, x.align);
  for (;;) {
    if (o > capacity - x.numel) return -1;
    const int64_t end = o + x.numel;
    int64_t k0 = o / S + 1;
    int64_t cut = -1;
    for (int64_t k = k0; k <= k0 + 1; ++k) {
      const int64_t boundary = k * S;
      if (boundary >= end) break;
      if ((boundary - o) % x.atom != 0) {
        cut = boundary;
        break;
      }
      if (S % x.atom == 0) break;  // every later boundary is on an atom edge too
    }
    if (cut < 0) return o;
    o = round_up(cut, x.align);
  }
}

bool place_all(const std::vector<TensorInfo>& ts, const std::vector<int>& order, int64_t m,
               int64_t S, std::vector<int64_t>* offsets) {
  int64_t capacity;
  if (!mul_ok(m, S, &capacity)) return false;
  int64_t cursor = 0;
  for (int t : order) {
    const TensorInfo& x = ts[t];
    // Quick reject: a tensor longer than 2S spans two consecutive boundaries,
    // which forces atom | S.
    if (x.numel > 2 * S && S % x.atom != 0) return false;
    int64_t o = earliest_offset(x, S, capacity, cursor);
    if (o < 0) return false;
    if (offsets) (*offsets)[t] = o;
    cursor = o + x.numel;
  }
  return true;
}

std::vector<int> order_for(const std::vector<TensorInfo>& ts, int policy) {
  std::vector<int> ord(ts.size());
  std::iota(ord.begin(), ord.end(), 0);
  if (policy == VSF_ORDER_BLOCK)
    std::stable_sort(ord.begin(), ord.end(), [&](int a, int b) { return ts[a].atom > ts[b].atom; });
  else if (policy == VSF_ORDER_SHAPE)
    std::stable_sort(ord.begin(), ord.end(),
                     [&](int a, int b) { return ts[a].numel > ts[b].numel; });
  return ord;
}

// Smallest feasible S for one order, or -1.
int64_t scan_S(const std::vector<TensorInfo>& ts, const std::vector<int>& order, int64_t m,
               int64_t g, int64_t real) {
  int64_t lb = round_up((real + m - 1) / m, g);
  // Everything aligned inside rank 0 always fits: an upper end for the scan.
  int64_t ub = 0;
  for (const TensorInfo& x : ts) ub += x.numel + x.align;
  ub = round_up(ub, g);
  for (int64_t S = lb; S <= std::max(lb, ub); S += g) {
    if (place_all(ts, order, m, S, nullptr)) return S;
  }
  return -1;
}

}  // namespace

vsf_status fail(vsf_status s, const std::string& msg) {
  g_last_error = msg;
  return s;
}

// Host-side check of the tables every kernel trusts: tensors inside the
// buffer and disjoint; each tensor's blocks inside its elements of the rank
// window (counted from the window start) and covering them exactly once.
vsf_status check_tables(const vsf_plan& plan) {
  const std::vector<TensorInfo>& ts = plan.tensors;
  std::vector<int> by_offset(ts.size());
  std::iota(by_offset.begin(), by_offset.end(), 0);
  std::sort(by_offset.begin(), by_offset.end(),
            [&](int a, int b) { return ts[a].offset < ts[b].offset; });
  int64_t end = 0;
  for (int t : by_offset) {
    if (ts[t].offset < end) return fail(VSF_ERR_STATE, "layout check: tensors overlap");
    end = ts[t].offset + ts[t].numel;
  }
  if (end > (int64_t)plan.m * plan.S) return fail(VSF_ERR_STATE, "layout check: past m * S");
  const int64_t wlo = (int64_t)plan.rank_begin * plan.S;
  std::vector<int64_t> covered(ts.size(), 0);
  for (const QBlock& b : plan.qblocks) {
    if (b.tensor < 0 || b.tensor >= (int)ts.size() || b.nrows < 1 || b.ncols < 1 ||
        (b.nrows > 1 && b.stride < b.ncols))
      return fail(VSF_ERR_STATE, "layout check: malformed block");
    const TensorInfo& x = ts[b.tensor];
    const int64_t first = b.base + wlo - x.offset;  // tensor element of the block start
    const int64_t last = first + (int64_t)(b.nrows - 1) * b.stride + b.ncols;  // one past
    if (first < x.lo || last > x.hi)
      return fail(VSF_ERR_STATE, "layout check: block outside its tensor's window");
    covered[b.tensor] += (int64_t)b.nrows * b.ncols;
  }
  for (size_t t = 0; t < ts.size(); ++t)
    if (covered[t] != ts[t].hi - ts[t].lo)
      return fail(VSF_ERR_STATE, "layout check: blocks do not cover tensor " + std::to_string(t));
  return VSF_OK;
}

// Quantisation-block tables, tile maps and the workspace layout for the rank
// window [r0, r1). Only blocks inside the window are listed (no block
// crosses a rank boundary: RaggedShard's Non-Sharded Block rule for row and
// tile atoms; element chunks start on g_coll multiples, as do offsets and
// S). Buffer elements are counted from the window start r0 * S.
static vsf_status build_tables_for(vsf_plan* plan, int32_t r0, int32_t r1) {
  const int n = plan->n;
  const int64_t chunk = tma_chunk_elems(plan->tma_warps);
  const int64_t g_coll = plan->g_coll;
  const int64_t wlo = (int64_t)r0 * plan->S, whi = (int64_t)r1 * plan->S;
  plan->rank_begin = r0;
  plan->rank_end = r1;
  plan->total = whi - wlo;
  plan->qblocks.clear();
  plan->big_blocks.clear();
  plan->tma_blocks.clear();
  plan->tma_tiles.clear();
  plan->tile_maps.clear();
  plan->small_blocks.clear();
  plan->max_big_elems = 0;
  plan->max_tma_elems = 0;
  double tma_sum = 0.0, tma_sumsq = 0.0;
  std::vector<TensorInfo>& ts = plan->tensors;
  int64_t real = 0;
  for (TensorInfo& x : ts) {
    x.lo = std::min(x.numel, std::max<int64_t>(0, wlo - x.offset));
    x.hi = std::max(x.lo, std::min(x.numel, whi - x.offset));
    real += x.hi - x.lo;
  }
  plan->real = real;

  // Quantisation blocks, tensor order ([VSF] case study › 8-bit Adam).
  for (int t = 0; t < n; ++t) {
    const TensorInfo& x = ts[t];
    if (x.lo >= x.hi) continue;  // no element inside the window
    const int64_t off = x.offset - wlo;  // window element of the tensor's element 0
    // Rows inside the window: whole stripes for row and tile atoms.
    const int64_t row_lo = x.lo / x.cols, row_hi = x.hi / x.cols;
    // Tile tensors whose full tiles go to the bulk-copy kernel as 2-D tensor
    // copies: tile width a power of two in [32, 256], k = 256 / width tiles
    // per work unit (one copy box of 256 columns), whole boxes of rows per
    // tile, 16-element aligned rows and window offset.
    int map = -1;
    int64_t k = 1;
    if (x.gran == VSF_GRAN_TILE && (int)plan->tile_maps.size() < kMaxTileMaps) {
      const int64_t bc = x.tile_cols, br = x.block_rows;
      if (bc >= 32 && bc <= 256 && (bc & (bc - 1)) == 0) {
        k = std::min<int64_t>(256 / bc, kMaxUnitTiles);
        const int64_t box_cols = k * bc;
        const int64_t box_rows = std::min<int64_t>(br, chunk / box_cols);
        const int64_t map_off = off + row_lo * x.cols;
        if (box_rows >= 1 && box_rows <= 256 && br % box_rows == 0 && x.cols % 16 == 0 &&
            map_off % 16 == 0 && x.cols >= box_cols) {
          TileMapInfo mi;
          mi.tensor = t;
          mi.tile_cols = (int32_t)bc;
          mi.k = (int32_t)k;
          mi.box_cols = (int32_t)box_cols;
          mi.box_rows = (int32_t)box_rows;
          mi.rows = row_hi - row_lo;
          mi.cols = x.cols;
          mi.offset = map_off;
          map = (int)plan->tile_maps.size();
          plan->tile_maps.push_back(mi);
        }
      }
    }
    // Where a block goes: element chunks to the warp kernel; contiguous
    // blocks that start on 16 elements and hold a multiple of 16, and full
    // tiles grouped k at a time, to the bulk-copy (TMA) kernel; every other
    // row or tile block (ragged, unaligned, leftover) to the register kernel.
    enum Dest { kSmall, kTma, kTmaTile, kTmaTileMember, kRegister };
    auto add = [&](int64_t base, int64_t nr, int64_t nc, int64_t st, Dest dest, int64_t r,
                   int64_t c) {
      QBlock b{};
      b.base = base;
      b.nrows = (int32_t)nr;
      b.ncols = (int32_t)nc;
      b.stride = (int32_t)st;
      b.tensor = t;
      b.tx = -1;
      b.ty = -1;
      const int32_t q = (int32_t)plan->qblocks.size();
      if (dest == kTmaTile || dest == kTmaTileMember) {
        b.tx = (int32_t)c;
        b.ty = (int32_t)(r - row_lo);  // row inside the tile map
      }
      if (dest == kSmall) {
        plan->small_blocks.push_back(q);
      } else if (dest == kTma || dest == kTmaTile) {
        plan->tma_blocks.push_back(q);
        plan->tma_tiles.push_back(dest == kTmaTile ? (int32_t)k : 1);
        const int64_t unit = nr * nc * (dest == kTmaTile ? k : 1);
        plan->max_tma_elems = std::max(plan->max_tma_elems, unit);
        tma_sum += (double)unit;
        tma_sumsq += (double)unit * (double)unit;
      } else if (dest == kRegister) {
        plan->big_blocks.push_back(q);
        plan->max_big_elems = std::max(plan->max_big_elems, nr * nc);
      }
      plan->qblocks.push_back(b);
    };
    if (x.gran == VSF_GRAN_ELEM) {
      if (g_coll > INT32_MAX) return fail(VSF_ERR_OVERFLOW, "g_coll too large for element-granular blocks");
      for (int64_t e = x.lo; e < x.hi; e += g_coll) {
        const int64_t len = std::min(g_coll, x.numel - e);
        add(off + e, 1, len, len, kSmall, 0, e);
      }
    } else if (x.gran == VSF_GRAN_ROWS) {
      for (int64_t r = row_lo; r < row_hi; r += x.block_rows) {
        const int64_t nr = std::min(x.block_rows, x.rows - r);
        // a whole-row block is contiguous: one row of nr*cols elements
        if (nr * x.cols > INT32_MAX)
          return fail(VSF_ERR_OVERFLOW, "quantisation block larger than 2^31 elements");
        const int64_t base = off + r * x.cols, len = nr * x.cols;
        add(base, 1, len, len, base % 16 == 0 && len % 16 == 0 ? kTma : kRegister, r, 0);
      }
    } else {
      if (x.cols > INT32_MAX || x.rows > INT32_MAX)
        return fail(VSF_ERR_OVERFLOW, "tile tensor dimension beyond 2^31");
      const int64_t tc = x.tile_cols;
      for (int64_t r = row_lo; r < row_hi; r += x.block_rows) {
        const int64_t nr = std::min(x.block_rows, x.rows - r);
        const int64_t full = nr == x.block_rows ? x.cols / tc : 0;  // full tiles in the stripe
        const int64_t grouped = map >= 0 ? full / k * k : 0;       // of them, in whole units
        for (int64_t c = 0, i = 0; c < x.cols; c += tc, ++i) {
          const int64_t nc = std::min(tc, x.cols - c);
          const Dest dest = i < grouped ? (i % k == 0 ? kTmaTile : kTmaTileMember) : kRegister;
          add(off + r * x.cols + c, nr, nc, x.cols, dest, r, c);
        }
      }
    }
  }

  plan->tma_unit_mean = tma_sum > 0.0 ? tma_sumsq / tma_sum : 0.0;
  const vsf_status checked = check_tables(*plan);
  if (checked != VSF_OK) return checked;

  // Device workspace layout (256-byte aligned sections).
  DeviceLayout& L = plan->layout;
  L = DeviceLayout();
  size_t cur = 0;
  auto section = [&](size_t bytes) {
    size_t at = (cur + 255) / 256 * 256;
    cur = at + bytes;
    return at;
  };
  L.tensor_off = section(sizeof(int64_t) * n);
  L.tensor_lo = section(sizeof(int64_t) * n);
  L.tensor_hi = section(sizeof(int64_t) * n);
  L.qblocks = section(sizeof(QBlock) * plan->qblocks.size());
  L.big = section(sizeof(int32_t) * std::max<size_t>(1, plan->big_blocks.size()));
  L.small = section(sizeof(int32_t) * std::max<size_t>(1, plan->small_blocks.size()));
  L.tma = section(sizeof(int32_t) * std::max<size_t>(1, plan->tma_blocks.size()));
  L.tma_k = section(sizeof(int32_t) * std::max<size_t>(1, plan->tma_tiles.size()));
  L.tma_start = section(sizeof(int32_t) * (kMaxCopyGrid + 1));
  L.error = section(16);
  L.spans = section(sizeof(CopySpan) * (kMaxCopyGrid + 1));
  L.partials = section(sizeof(double) * kMaxCopyGrid);
  L.bytes = (cur + 255) / 256 * 256;
  return VSF_OK;
}

// The tables with the wide bulk-copy chunk; if every work unit is small,
// again with the narrow one. Tile copy boxes follow the chunk size, so a
// smaller chunk can only move tile units to the register kernel (a stripe
// height the shorter box does not divide), never enlarge one; if it moves
// any, the wide tables are rebuilt and kept.
vsf_status build_tables(vsf_plan* plan, int32_t r0, int32_t r1) {
  if (plan->forced_warps != 0) {
    plan->tma_warps = plan->forced_warps;
    return build_tables_for(plan, r0, r1);
  }
  plan->tma_warps = kTmaWideWarps;
  vsf_status st = build_tables_for(plan, r0, r1);
  if (st != VSF_OK || plan->max_tma_elems == 0 || plan->max_tma_elems > kTmaNarrowMaxUnit)
    return st;
  const size_t wide_units = plan->tma_blocks.size();
  plan->tma_warps = kTmaNarrowWarps;
  st = build_tables_for(plan, r0, r1);
  if (st != VSF_OK || plan->tma_blocks.size() == wide_units) return st;
  plan->tma_warps = kTmaWideWarps;
  return build_tables_for(plan, r0, r1);
}


const char* last_error() { return g_last_error.c_str(); }

}  // namespace vsf

using vsf::fail;

extern "C" {

vsf_status vsf_plan_create(const vsf_tensor_desc* descs, int32_t n, int32_t m, int64_t g_coll,
                           int32_t order, vsf_plan** out) {
  vsf::Range nvtx_range("vsf_plan_create");
  const auto t0 = std::chrono::steady_clock::now();
  if (out == nullptr) return fail(VSF_ERR_ARG, "vsf_plan_create: out is NULL");
  *out = nullptr;
  if (descs == nullptr || n < 1) return fail(VSF_ERR_ARG, "vsf_plan_create: no tensors");
  if (m < 1) return fail(VSF_ERR_ARG, "vsf_plan_create: m must be >= 1");
  if (g_coll < 1) return fail(VSF_ERR_ARG, "vsf_plan_create: g_coll must be >= 1");
  if (order < VSF_ORDER_DEFAULT || order > VSF_ORDER_BEST3)
    return fail(VSF_ERR_ARG, "vsf_plan_create: unknown order policy");

  std::vector<vsf::TensorInfo> ts(n);
  int64_t real = 0;
  for (int t = 0; t < n; ++t) {
    const vsf_tensor_desc& d = descs[t];
    vsf::TensorInfo& x = ts[t];
    if (d.ndim < 1 || d.ndim > 8)
      return fail(VSF_ERR_ARG, "tensor " + std::to_string(t) + ": ndim must be 1..8");
    int64_t rows = 1;
    for (int k = 0; k < d.ndim; ++k)
      if (d.shape[k] < 1) return fail(VSF_ERR_ARG, "tensor " + std::to_string(t) + ": empty dim");
    for (int k = 0; k + 1 < d.ndim; ++k)
      if (!vsf::mul_ok(rows, d.shape[k], &rows)) return fail(VSF_ERR_OVERFLOW, "rows overflow");
    x.ndim = d.ndim;
    for (int k = 0; k < 8; ++k) x.shape[k] = k < d.ndim ? d.shape[k] : 1;
    x.rows = rows;
    x.cols = d.shape[d.ndim - 1];
    if (!vsf::mul_ok(x.rows, x.cols, &x.numel)) return fail(VSF_ERR_OVERFLOW, "numel overflow");
    x.gran = d.gran;
    x.block_rows = d.block_rows;
    x.tile_cols = d.tile_cols;
    if (x.gran == VSF_GRAN_ELEM) {
      x.atom = 1;
    } else if (x.gran == VSF_GRAN_ROWS || x.gran == VSF_GRAN_TILE) {
      if (x.block_rows < 1)
        return fail(VSF_ERR_ARG, "tensor " + std::to_string(t) + ": block_rows must be >= 1");
      if (x.gran == VSF_GRAN_TILE && x.tile_cols < 1)
        return fail(VSF_ERR_ARG, "tensor " + std::to_string(t) + ": tile_cols must be >= 1");
      if (!vsf::mul_ok(x.block_rows, x.cols, &x.atom)) return fail(VSF_ERR_OVERFLOW, "atom");
    } else {
      return fail(VSF_ERR_ARG, "tensor " + std::to_string(t) + ": unknown granularity");
    }
    const int64_t q = g_coll / vsf::gcd64(g_coll, x.atom);
    if (!vsf::mul_ok(q, x.atom, &x.align)) return fail(VSF_ERR_OVERFLOW, "alignment overflow");
    if (real > INT64_MAX - x.numel) return fail(VSF_ERR_OVERFLOW, "total overflow");
    real += x.numel;
  }
  // Headroom so that offsets + spans + alignment never overflow.
  if (real > (INT64_MAX >> 4)) return fail(VSF_ERR_OVERFLOW, "too many elements");

  int64_t best_S = -1;
  int used = VSF_ORDER_DEFAULT;
  const int first = order == VSF_ORDER_BEST3 ? VSF_ORDER_DEFAULT : order;
  const int last = order == VSF_ORDER_BEST3 ? VSF_ORDER_SHAPE : order;
  for (int p = first; p <= last; ++p) {
    int64_t S = vsf::scan_S(ts, vsf::order_for(ts, p), m, g_coll, real);
    if (S >= 0 && (best_S < 0 || S < best_S)) {
      best_S = S;
      used = p;
    }
  }
  if (best_S < 0) return fail(VSF_ERR_INFEASIBLE, "no feasible layout");

  std::vector<int64_t> offsets(n);
  vsf::place_all(ts, vsf::order_for(ts, used), m, best_S, &offsets);

  auto* plan = new vsf_plan();
  plan->n = n;
  plan->m = m;
  plan->g_coll = g_coll;
  plan->S = best_S;
  plan->order_used = used;
  for (int t = 0; t < n; ++t) ts[t].offset = offsets[t];
  plan->tensors = ts;
  const vsf_status st = vsf::build_tables(plan, 0, m);
  if (st != VSF_OK) {
    delete plan;
    return st;
  }
  plan->plan_seconds =
      std::chrono::duration<double>(std::chrono::steady_clock::now() - t0).count();
  *out = plan;
  return VSF_OK;
}

vsf_status vsf_plan_restrict(vsf_plan* plan, int32_t rank_begin, int32_t rank_end) {
  if (plan == nullptr) return fail(VSF_ERR_ARG, "vsf_plan_restrict: NULL plan");
  if (plan->uploaded) return fail(VSF_ERR_STATE, "vsf_plan_restrict: plan already uploaded");
  if (rank_begin < 0 || rank_end > plan->m || rank_begin >= rank_end)
    return fail(VSF_ERR_ARG, "vsf_plan_restrict: need 0 <= rank_begin < rank_end <= m");
  return vsf::build_tables(plan, rank_begin, rank_end);
}

vsf_status vsf_plan_set_bulk_warps(vsf_plan* plan, int32_t warps) {
  if (plan == nullptr) return fail(VSF_ERR_ARG, "vsf_plan_set_bulk_warps: NULL plan");
  if (plan->uploaded) return fail(VSF_ERR_STATE, "vsf_plan_set_bulk_warps: plan already uploaded");
  if (warps != 0 && warps != vsf::kTmaWideWarps && warps != vsf::kTmaNarrowWarps)
    return fail(VSF_ERR_ARG, "vsf_plan_set_bulk_warps: warps must be 0, 4 or 16");
  plan->forced_warps = warps;
  return vsf::build_tables(plan, plan->rank_begin, plan->rank_end);
}

void vsf_plan_destroy(vsf_plan* plan) { delete plan; }

namespace {
constexpr uint32_t kPlanMagic = 0x50465356u;  // "VSFP"
constexpr uint32_t kPlanVersion = 1;

// Fixed-size part of a serialized plan, then n descriptors, n offsets and
// the checksum of everything before it.
struct PlanHeader {
  uint32_t magic, version;
  int32_t n, m;
  int64_t g_coll;
  int32_t order, rank_begin, rank_end, forced_warps;
  int64_t S;
};

uint64_t fnv1a(const unsigned char* p, size_t len) {
  uint64_t h = 0xcbf29ce484222325ull;
  for (size_t i = 0; i < len; ++i) {
    h ^= p[i];
    h *= 0x100000001b3ull;
  }
  return h;
}

size_t plan_bytes(int32_t n) {
  return sizeof(PlanHeader) + (size_t)n * (sizeof(vsf_tensor_desc) + sizeof(int64_t)) +
         sizeof(uint64_t);
}
}  // namespace

vsf_status vsf_plan_serialize(const vsf_plan* plan, void* buf, size_t* bytes) {
  if (plan == nullptr || bytes == nullptr) return fail(VSF_ERR_ARG, "vsf_plan_serialize: NULL argument");
  const size_t need = plan_bytes(plan->n);
  if (buf == nullptr) {
    *bytes = need;
    return VSF_OK;
  }
  if (*bytes < need) {
    *bytes = need;
    return fail(VSF_ERR_ARG, "vsf_plan_serialize: buffer too small");
  }
  unsigned char* p = static_cast<unsigned char*>(buf);
  PlanHeader h;
  std::memset(&h, 0, sizeof(h));
  h.magic = kPlanMagic;
  h.version = kPlanVersion;
  h.n = plan->n;
  h.m = plan->m;
  h.g_coll = plan->g_coll;
  h.order = plan->order_used;
  h.rank_begin = plan->rank_begin;
  h.rank_end = plan->rank_end;
  h.forced_warps = plan->forced_warps;
  h.S = plan->S;
  std::memcpy(p, &h, sizeof(h));
  size_t at = sizeof(h);
  for (int t = 0; t < plan->n; ++t) {
    const vsf::TensorInfo& x = plan->tensors[t];
    vsf_tensor_desc d;
    std::memset(&d, 0, sizeof(d));
    d.ndim = x.ndim;
    d.gran = x.gran;
    for (int k = 0; k < x.ndim; ++k) d.shape[k] = x.shape[k];
    d.block_rows = x.block_rows;
    d.tile_cols = x.tile_cols;
    std::memcpy(p + at, &d, sizeof(d));
    at += sizeof(d);
  }
  for (int t = 0; t < plan->n; ++t) {
    std::memcpy(p + at, &plan->tensors[t].offset, sizeof(int64_t));
    at += sizeof(int64_t);
  }
  const uint64_t sum = fnv1a(p, at);
  std::memcpy(p + at, &sum, sizeof(sum));
  *bytes = need;
  return VSF_OK;
}

vsf_status vsf_plan_deserialize(const void* buf, size_t bytes, vsf_plan** out) {
  if (buf == nullptr || out == nullptr) return fail(VSF_ERR_ARG, "vsf_plan_deserialize: NULL argument");
  *out = nullptr;
  const unsigned char* p = static_cast<const unsigned char*>(buf);
  if (bytes < sizeof(PlanHeader)) return fail(VSF_ERR_ARG, "vsf_plan_deserialize: truncated");
  PlanHeader h;
  std::memcpy(&h, p, sizeof(h));
  if (h.magic != kPlanMagic) return fail(VSF_ERR_ARG, "vsf_plan_deserialize: not a serialized plan");
  if (h.version != kPlanVersion) return fail(VSF_ERR_ARG, "vsf_plan_deserialize: unknown version");
  if (h.n < 1 || h.n > vsf::kMaxTensors || bytes != plan_bytes(h.n))
    return fail(VSF_ERR_ARG, "vsf_plan_deserialize: size does not match the tensor count");
  const size_t body = bytes - sizeof(uint64_t);
  uint64_t sum;
  std::memcpy(&sum, p + body, sizeof(sum));
  if (sum != fnv1a(p, body)) return fail(VSF_ERR_ARG, "vsf_plan_deserialize: checksum mismatch");
  std::vector<vsf_tensor_desc> descs((size_t)h.n);
  std::vector<int64_t> offsets((size_t)h.n);
  size_t at = sizeof(h);
  std::memcpy(descs.data(), p + at, sizeof(vsf_tensor_desc) * descs.size());
  at += sizeof(vsf_tensor_desc) * descs.size();
  std::memcpy(offsets.data(), p + at, sizeof(int64_t) * offsets.size());
  if (h.order < VSF_ORDER_DEFAULT || h.order > VSF_ORDER_SHAPE)
    return fail(VSF_ERR_ARG, "vsf_plan_deserialize: bad order policy");
  vsf_plan* plan = nullptr;
  vsf_status st = vsf_plan_create(descs.data(), h.n, h.m, h.g_coll, h.order, &plan);
  if (st != VSF_OK) return st;
  if (plan->S != h.S) {
    vsf_plan_destroy(plan);
    return fail(VSF_ERR_STATE, "vsf_plan_deserialize: the planner gives another S for these inputs");
  }
  for (int t = 0; t < h.n; ++t)
    if (plan->tensors[t].offset != offsets[(size_t)t]) {
      vsf_plan_destroy(plan);
      return fail(VSF_ERR_STATE, "vsf_plan_deserialize: the planner gives other offsets for these inputs");
    }
  if (h.rank_begin != 0 || h.rank_end != h.m) st = vsf_plan_restrict(plan, h.rank_begin, h.rank_end);
  if (st == VSF_OK && h.forced_warps != 0) st = vsf_plan_set_bulk_warps(plan, h.forced_warps);
  if (st != VSF_OK) {
    vsf_plan_destroy(plan);
    return st;
  }
  *out = plan;
  return VSF_OK;
}

vsf_status vsf_plan_get_info(const vsf_plan* plan, vsf_plan_info* info) {
  if (plan == nullptr || info == nullptr) return fail(VSF_ERR_ARG, "NULL argument");
  std::memset(info, 0, sizeof(*info));
  info->S = plan->S;
  info->total = plan->total;
  info->real = plan->real;
  info->n_qblocks = (int64_t)plan->qblocks.size();
  info->n_tensors = plan->n;
  info->m = plan->m;
  info->g_coll = plan->g_coll;
  info->padding_ratio = 1.0 - (double)plan->real / (double)plan->total;
  info->plan_seconds = plan->plan_seconds;
  info->order_used = plan->order_used;
  info->bulk_warps = plan->tma_warps;
  info->n_bulk_units = (int64_t)plan->tma_blocks.size();
  info->n_register_blocks = (int64_t)plan->big_blocks.size();
  info->n_element_chunks = (int64_t)plan->small_blocks.size();
  info->rank_begin = plan->rank_begin;
  info->rank_end = plan->rank_end;
  info->bulk_cluster = plan->uploaded ? plan->tma_cluster : 0;
  return VSF_OK;
}

vsf_status vsf_plan_offsets(const vsf_plan* plan, int64_t* offsets) {
  if (plan == nullptr || offsets == nullptr) return fail(VSF_ERR_ARG, "NULL argument");
  for (int t = 0; t < plan->n; ++t) offsets[t] = plan->tensors[t].offset;
  return VSF_OK;
}

vsf_status vsf_plan_qblocks(const vsf_plan* plan, int32_t* tensor, int64_t* base, int64_t* nrows,
                            int64_t* ncols, int64_t* stride) {
  if (plan == nullptr) return fail(VSF_ERR_ARG, "NULL plan");
  for (size_t q = 0; q < plan->qblocks.size(); ++q) {
    const vsf::QBlock& b = plan->qblocks[q];
    const vsf::TensorInfo& x = plan->tensors[b.tensor];
    // ROWS blocks are stored as one contiguous row; report them as rows x cols.
    const bool rows_block = x.gran == VSF_GRAN_ROWS;
    if (tensor) tensor[q] = b.tensor;
    if (base) base[q] = b.base;
    if (nrows) nrows[q] = rows_block ? b.ncols / x.cols : b.nrows;
    if (ncols) ncols[q] = rows_block ? x.cols : b.ncols;
    if (stride) stride[q] = rows_block ? x.cols : b.stride;
  }
  return VSF_OK;
}

vsf_status vsf_plan_rank_slices(const vsf_plan* plan, int32_t rank, int32_t capacity,
                                int32_t* count, int32_t* tensor, int64_t* elem_begin,
                                int64_t* elem_end, int64_t* atom_begin, int64_t* atom_end) {
  if (plan == nullptr || count == nullptr) return fail(VSF_ERR_ARG, "NULL argument");
  if (rank < 0 || rank >= plan->m) return fail(VSF_ERR_ARG, "rank out of range");
  std::vector<int> by_offset(plan->n);
  std::iota(by_offset.begin(), by_offset.end(), 0);
  std::sort(by_offset.begin(), by_offset.end(), [&](int a, int b) {
    return plan->tensors[a].offset < plan->tensors[b].offset;
  });
  const int64_t lo = (int64_t)rank * plan->S, hi = lo + plan->S;
  int32_t k = 0;
  for (int t : by_offset) {
    const vsf::TensorInfo& x = plan->tensors[t];
    const int64_t b = std::max(lo, x.offset), e = std::min(hi, x.offset + x.numel);
    if (b >= e) continue;
    if (k < capacity) {
      if (tensor) tensor[k] = t;
      if (elem_begin) elem_begin[k] = b - x.offset;
      if (elem_end) elem_end[k] = e - x.offset;
      if (atom_begin) atom_begin[k] = (b - x.offset) / x.atom;
      if (atom_end) atom_end[k] = (e - x.offset + x.atom - 1) / x.atom;
    }
    ++k;
  }
  *count = k;
  return VSF_OK;
}

vsf_status vsf_plan_device_error_offset(const vsf_plan* plan, size_t* offset) {
  if (plan == nullptr || offset == nullptr) return fail(VSF_ERR_ARG, "NULL argument");
  *offset = plan->layout.error;
  return VSF_OK;
}

vsf_status vsf_plan_views(const vsf_plan* plan, const void* packed, int32_t elem_bytes,
                          void** views) {
  if (plan == nullptr || packed == nullptr || views == nullptr)
    return fail(VSF_ERR_ARG, "vsf_plan_views: NULL argument");
  if (elem_bytes != 1 && elem_bytes != 2 && elem_bytes != 4)
    return fail(VSF_ERR_ARG, "vsf_plan_views: elem_bytes must be 1, 2 or 4");
  if (plan->rank_begin != 0 || plan->rank_end != plan->m)
    return fail(VSF_ERR_STATE, "vsf_plan_views: whole tensors live only in an unrestricted plan");
  for (int t = 0; t < plan->n; ++t)
    views[t] = const_cast<char*>(static_cast<const char*>(packed)) +
               plan->tensors[t].offset * (int64_t)elem_bytes;
  return VSF_OK;
}

size_t vsf_plan_workspace_bytes(const vsf_plan* plan) {
  return plan == nullptr ? 0 : plan->layout.bytes;
}

const char* vsf_status_string(vsf_status s) {
  switch (s) {
    case VSF_OK: return "ok";
    case VSF_ERR_ARG: return "invalid argument";
    case VSF_ERR_INFEASIBLE: return "no feasible layout";
    case VSF_ERR_OVERFLOW: return "size overflow";
    case VSF_ERR_ALIGN: return "pointer not 16-byte aligned";
    case VSF_ERR_CUDA: return "CUDA error";
    case VSF_ERR_STATE: return "call out of order";
    default: return "unknown status";
  }
}

const char* vsf_last_error(void) { return vsf::last_error(); }

}  // extern "C"
