// vsf_internal.h — plan representation shared by the host planner
// (plan.cpp) and the kernels (vsf_kernels.cu) inside libvsf. Not installed.
#pragma once

#include <cstddef>
#include <cstdint>
#include <mutex>

#include <nvtx3/nvToolsExt.h>
#include <string>
#include <vector>

#include "vsf.h"

namespace vsf {

// Most per-tensor device pointers one pack / unpack launch takes by value
// (16 KB of kernel parameters).
constexpr int kMaxTensors = 2048;
// Upper bound of the copy grid, which fixes the workspace size before the
// device is known.
constexpr int kMaxCopyGrid = 4096;

// Bulk-copy (TMA) AdamW kernel geometry. Each consumer thread takes two
// 8-element groups of a ring chunk, so a chunk holds warps * 512 elements.
// Two shapes, chosen per plan: wide (16 consumer warps, one CTA per SM) for
// plans with large work units, narrow (4 consumer warps, four CTAs per SM)
// when every unit has at most kTmaNarrowMaxUnit elements. Small units leave a
// single pipeline per SM idle while its consumers wait for the block maxima;
// four pipelines per SM overlap those waits. The bound keeps the narrow
// shape's clusters small: 4 CTAs on each of 152 SMs, each cluster holding
// one unit's gradient and codes (4 bytes an element for bf16 gradients) in
// L2 between the two passes, keep 608 * 4 * 48 Ki = 114 MB in flight at the
// bound in clusters of 1, and half that in clusters of 2, which the bulk
// kernel's L2 rule (half the L2) then picks.
constexpr int kTmaGroups = 2;
constexpr int kTmaWideWarps = 16;
constexpr int kTmaNarrowWarps = 4;
constexpr int64_t kTmaNarrowMaxUnit = 48 * 1024;
constexpr int tma_chunk_elems(int warps) { return warps * 32 * 8 * kTmaGroups; }

// One quantisation block as the kernels see it: a row-major region.
struct QBlock {
  int64_t base;    // buffer element of the first element
  int32_t nrows;   // rows in the block
  int32_t ncols;   // elements per row
  int32_t stride;  // elements between row starts
  int32_t tensor;
  int32_t tx, ty;  // tiles read by 2-D tensor copies: column and row in the tensor; else -1
};
static_assert(sizeof(QBlock) == 32, "QBlock is a 32-byte device record");

// Where one CTA of the copy grid starts in the concatenation of the real
// elements the plan covers (tensor order; each tensor's [lo, hi) range).
struct CopySpan {
  int32_t tensor;
  int32_t pad;
  int64_t elem;
};

// Tile tensors whose full tiles the bulk-copy kernel reads with 2-D tensor
// copies (one tensor map per array and tensor, encoded per call).
// A work unit of that kernel is k adjacent full tiles of one stripe, read
// together as one box of k * tile_cols (<= 256) columns.
constexpr int kMaxTileMaps = 16;
constexpr int kMaxUnitTiles = 8;
struct TileMapInfo {
  int32_t tensor;
  int32_t tile_cols, k;        // tile width; tiles per work unit
  int32_t box_cols, box_rows;  // one copy = box_rows rows of box_cols = k * tile_cols elements
  int64_t rows, cols, offset;  // the 2-D view (rows inside the plan's window) in the buffer
};

struct TensorInfo {
  int32_t ndim;
  int64_t shape[8];
  int64_t rows, cols, numel;
  int32_t gran;
  int64_t block_rows, tile_cols;
  int64_t atom, align;
  int64_t offset;  // global buffer element of the tensor's first element
  int64_t lo, hi;  // the tensor's elements inside the plan's rank window
};

struct DeviceLayout {
  size_t tensor_off = 0;                    // int64[n]: offset minus the window start
  size_t tensor_lo = 0, tensor_hi = 0;      // int64[n]: element range inside the window
  size_t qblocks = 0;                       // QBlock[n_qblocks]
  size_t big = 0, small = 0, tma = 0;       // int32 lists of block indices
  size_t tma_k = 0;                         // int32 tiles per TMA work unit
  size_t tma_start = 0;                     // int32[kMaxCopyGrid + 1]: first unit of each cluster
  size_t error = 0;                         // uint32 device error word
  size_t spans = 0;                         // CopySpan[kMaxCopyGrid + 1]
  size_t partials = 0;                      // double[kMaxCopyGrid]
  size_t bytes = 0;
};

}  // namespace vsf

struct vsf_plan {
  int32_t n = 0, m = 0;
  int64_t g_coll = 0, S = 0, total = 0, real = 0;  // total, real: inside the rank window
  int32_t order_used = 0;
  // Rank window [rank_begin, rank_end): buffers passed to the per-step calls
  // hold elements [rank_begin * S, rank_end * S) of the planned buffer.
  int32_t rank_begin = 0, rank_end = 0;
  double plan_seconds = 0.0;
  std::vector<vsf::TensorInfo> tensors;
  std::vector<vsf::QBlock> qblocks;
  std::vector<int32_t> big_blocks;    // ROWS / TILE blocks: register block kernel
  std::vector<int32_t> tma_blocks;    // TMA kernel work units: first block of each
  std::vector<int32_t> tma_tiles;     // tiles per unit (1 for a contiguous block)
  std::vector<vsf::TileMapInfo> tile_maps;
  std::vector<int32_t> small_blocks;  // ELEM chunks: warp kernel
  int64_t max_big_elems = 0;
  int64_t max_tma_elems = 0;
  // element-weighted mean unit size of the TMA units: sum n^2 / sum n (the
  // size of the unit an average element belongs to)
  double tma_unit_mean = 0.0;
  int tma_warps = vsf::kTmaWideWarps;  // shape of the bulk-copy kernel (consumer warps)
  int forced_warps = 0;                // vsf_plan_set_bulk_warps: 0 = the planner's choice
  vsf::DeviceLayout layout;

  // Set by vsf_plan_upload.
  bool uploaded = false;
  unsigned char* d_ws = nullptr;
  int device = -1;
  int sm_count = 0;
  int copy_grid = 0;
  int adam_cluster = 1;
  int adam_clusters = 0;
  int tma_cluster = 1;
  int tma_clusters = 0;
  std::vector<unsigned char> upload_image;  // host source of the last upload copy
  // Muon's second stream and its fork/join events, created at upload on the
  // plan's device (muon.cu owns the type and frees it).
  void* muon_lanes = nullptr;
  void (*muon_lanes_free)(void*) = nullptr;
  // Tensor maps of the tile tensors, encoded for the last pointers seen.
  mutable std::mutex maps_mu;
  mutable std::vector<unsigned char> maps_blob;  // kernel-parameter image
  mutable const void* maps_key[5] = {nullptr, nullptr, nullptr, nullptr, nullptr};
  mutable int maps_dtype = -1;

  vsf_plan() = default;
  vsf_plan(const vsf_plan&) = delete;
  vsf_plan& operator=(const vsf_plan&) = delete;
  ~vsf_plan() {
    if (muon_lanes_free != nullptr) muon_lanes_free(muon_lanes);
  }
};

namespace vsf {
// A named host range around one ABI call, for profilers' timelines (NVTX v3,
// header only; without an attached tool each push and pop is a no-op call).
struct Range {
  explicit Range(const char* name) { nvtxRangePushA(name); }
  ~Range() { nvtxRangePop(); }
  Range(const Range&) = delete;
  Range& operator=(const Range&) = delete;
};
vsf_status fail(vsf_status s, const std::string& msg);
// Creates Muon's second stream and its events on the current device (once
// per plan; muon.cu).
vsf_status muon_lanes_create(vsf_plan* plan);
vsf_status build_tables(vsf_plan* plan, int32_t r0, int32_t r1);
}  // namespace vsf
