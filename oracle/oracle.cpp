// oracle.cpp — TEST INFRASTRUCTURE. The plain, slow, single-threaded CPU oracle
// of the shard-step path (layout plan, copy-in, group grad norm and scale,
// block-wise 8-bit AdamW, copy-out).
//
// Only the test suite, the package smoke check and the benchmark's CPU-baseline
// leg may load this library. The CUDA library never includes, links or calls
// it, and this file includes nothing from that library: every type and loop
// below is its own.
//
// Sources, cited by page title and section:
//   [VSF]  "veScale-FSDP: Flexible and High-Performance FSDP at Scale
//          (MLSys 2026)" summary page.
//          - 核心方法 › RaggedShard: atomic blocks (element / row / 2-D block),
//            uneven block counts per device.
//          - 核心方法 › Grouped communication (Algorithm 1): minimum uniform
//            per-device size S under Non-Sharded Block, Contiguous Tensor
//            Memory and Balanced Load; tensor order (default / block size /
//            shape); placement; padding only between tensors, offsets aligned
//            to lcm(g_coll, block size).
//          - 核心方法 › Distributed Buffer: fused group ops (scale, copy) over
//            one global buffer.
//          - 结构感知训练 case study › 8-bit Adam: per-block quantisation that
//            stays local because blocks are never split across devices.
//   [FSDP] "FSDP" concept page › 关键观察: copy-in / copy-out around the
//          collective buffer.
// The pages define no quantiser and no AdamW op order. The readings used here
// (each marked "reading:") are: int8 m with symmetric per-block absmax, uint8
// v with per-block max, AdamW beta1=0.9, beta2=0.999, eps=1e-8, lr=1e-3,
// decoupled weight decay 0.01 with bias correction, round half to even, and
// the fp32 op order written out in adam_element().
//
// Parity status: layout, copy-in/out, grad norm and the fp32-state AdamW are
// pinned by the tests (invariants, brute force, closed forms, torch's AdamW),
// the tensor orders through the offsets they produce. The 8-bit
// requantisation is pinned only through its own properties and the
// first-step closed form, because the pages print no quantised values. A
// mutation test plants one mistake at a time into a copy of this file, and
// every one of them must fail a pin.
//
// Build: g++ -O2 -std=c++17 -ffp-contract=off (no FMA contraction: every fp32
// operation below rounds once, in the order written).

#include <algorithm>
#include <cfenv>
#include <cmath>
#include <cstdint>
#include <cstring>
#include <numeric>
#include <vector>

namespace {

enum { GRAN_ELEM = 0, GRAN_ROWS = 1, GRAN_TILE = 2 };
enum { ORDER_DEFAULT = 0, ORDER_BLOCK = 1, ORDER_SHAPE = 2, ORDER_BEST3 = 3 };

struct Tensor {
  int64_t rows = 0, cols = 0, numel = 0;
  int gran = GRAN_ELEM;
  int64_t block_rows = 0, tile_cols = 0;
  int64_t block = 1;  // shard atom in elements
  int64_t align = 1;  // lcm(g_coll, block)
};

int64_t gcd_i64(int64_t a, int64_t b) {
  while (b != 0) {
    int64_t t = a % b;
    a = b;
    b = t;
  }
  return a;
}

// Returns -1 on overflow.
int64_t lcm_i64(int64_t a, int64_t b) {
  int64_t g = gcd_i64(a, b);
  int64_t q = a / g;
  if (q != 0 && b > INT64_MAX / q) return -1;
  return q * b;
}

int64_t align_up(int64_t x, int64_t a) { return (x + a - 1) / a * a; }

// Shard atom of a tensor ([VSF] 核心方法 › RaggedShard): one element, or
// block_rows whole rows. reading: a 2-D block (block_rows x tile_cols) on
// row-major storage shards by block_rows-row stripes, so its atom is the
// stripe; the tile only sets the quantisation block.
bool make_tensors(int n, const int64_t* rows, const int64_t* cols, const int32_t* gran,
                  const int64_t* block_rows, const int64_t* tile_cols, int64_t g_coll,
                  std::vector<Tensor>& out) {
  if (n <= 0 || g_coll <= 0) return false;
  out.assign(n, Tensor());
  for (int t = 0; t < n; ++t) {
    Tensor& x = out[t];
    x.rows = rows[t];
    x.cols = cols[t];
    x.gran = gran[t];
    if (x.rows <= 0 || x.cols <= 0) return false;
    if (x.cols > INT64_MAX / x.rows) return false;
    x.numel = x.rows * x.cols;
    if (x.gran == GRAN_ELEM) {
      x.block = 1;
    } else if (x.gran == GRAN_ROWS || x.gran == GRAN_TILE) {
      x.block_rows = block_rows[t];
      if (x.block_rows <= 0) return false;
      if (x.gran == GRAN_TILE) {
        x.tile_cols = tile_cols[t];
        if (x.tile_cols <= 0) return false;
      }
      if (x.cols > INT64_MAX / x.block_rows) return false;
      x.block = x.block_rows * x.cols;
    } else {
      return false;
    }
    x.align = lcm_i64(g_coll, x.block);
    if (x.align <= 0) return false;
  }
  return true;
}

// Places the tensors in `order` one after another, each at the earliest
// offset that is a multiple of its alignment and that no rank boundary k*S
// cuts inside one of its atoms ([VSF] 核心方法 › Algorithm 1: Non-Sharded
// Block, Contiguous Tensor Memory, padding only between tensors). Returns
// false if the last tensor would end past m*S.
bool place(const std::vector<Tensor>& ts, const std::vector<int>& order, int64_t m, int64_t S,
           std::vector<int64_t>& offsets) {
  if (S > INT64_MAX / m) return false;
  const int64_t capacity = m * S;
  int64_t cursor = 0;
  offsets.assign(ts.size(), -1);
  for (int t : order) {
    const Tensor& x = ts[t];
    int64_t o = align_up(cursor, x.align);
    for (;;) {
      if (o > capacity - x.numel) return false;
      int64_t cut = -1;
      for (int64_t k = o / S + 1; k * S < o + x.numel; ++k) {
        if ((k * S - o) % x.block != 0) {
          cut = k * S;
          break;
        }
      }
      if (cut < 0) break;
      o = align_up(cut, x.align);
    }
    offsets[t] = o;
    cursor = o + x.numel;
  }
  return true;
}

// Lower bound on S: the balanced share of the real elements, rounded up to
// the collective unit ([VSF] Algorithm 1, Balanced Load).
int64_t lower_bound_S(const std::vector<Tensor>& ts, int64_t m, int64_t g_coll) {
  int64_t total = 0;
  for (const Tensor& x : ts) total += x.numel;
  return align_up((total + m - 1) / m, g_coll);
}

// Any S at least this large holds every tensor, aligned, inside rank 0.
int64_t feasible_bound_S(const std::vector<Tensor>& ts, int64_t g_coll) {
  int64_t s = 0;
  for (const Tensor& x : ts) s += x.numel + x.align;
  return align_up(s, g_coll);
}

// reading: Algorithm 1's objective is the smallest S that is a multiple of
// g_coll; feasibility is not monotone in S, so every candidate from the lower
// bound upward is tried in turn.
int64_t min_S_for_order(const std::vector<Tensor>& ts, const std::vector<int>& order, int64_t m,
                        int64_t g_coll, std::vector<int64_t>& offsets) {
  const int64_t lo = lower_bound_S(ts, m, g_coll);
  const int64_t hi = feasible_bound_S(ts, g_coll);
  for (int64_t S = lo; S <= std::max(lo, hi); S += g_coll) {
    if (place(ts, order, m, S, offsets)) return S;
  }
  return -1;
}

// Tensor orders of [VSF] Algorithm 1's first step. reading: "by block size"
// and "by shape" sort by atom size and by element count, descending, ties by
// input position.
std::vector<int> make_order(const std::vector<Tensor>& ts, int policy) {
  std::vector<int> ord(ts.size());
  std::iota(ord.begin(), ord.end(), 0);
  if (policy == ORDER_BLOCK) {
    std::stable_sort(ord.begin(), ord.end(),
                     [&](int a, int b) { return ts[a].block > ts[b].block; });
  } else if (policy == ORDER_SHAPE) {
    std::stable_sort(ord.begin(), ord.end(),
                     [&](int a, int b) { return ts[a].numel > ts[b].numel; });
  }
  return ord;
}

// ---------------------------------------------------------------- AdamW

struct AdamConsts {
  float b1, omb1, b2, omb2, eps_hat, decay, alpha;
};

// reading: the host-side constants of step t, each computed in double and
// rounded once to fp32; beta^t is t repeated multiplications. The update is
// the Adam paper's efficient form (Kingma & Ba, "Adam: A Method for
// Stochastic Optimization", end of section 2): alpha_t = lr sqrt(1-b2^t) /
// (1-b1^t) and eps_hat = eps sqrt(1-b2^t), which equals the bias-corrected
// update lr * mhat / (sqrt(vhat) + eps) in exact arithmetic.
AdamConsts adam_consts(double lr, double beta1, double beta2, double eps, double wd, int t) {
  double p1 = 1.0, p2 = 1.0;
  for (int i = 0; i < t; ++i) {
    p1 *= beta1;
    p2 *= beta2;
  }
  const double bc2s = std::sqrt(1.0 - p2);
  AdamConsts k;
  k.b1 = (float)beta1;
  k.omb1 = (float)(1.0 - beta1);
  k.b2 = (float)beta2;
  k.omb2 = (float)(1.0 - beta2);
  k.eps_hat = (float)(eps * bc2s);
  k.decay = (float)(1.0 - lr * wd);
  k.alpha = (float)(lr * bc2s / (1.0 - p1));
  return k;
}

// One AdamW element update with decoupled weight decay and bias correction.
// reading: this exact fp32 op order, every operation rounded once.
inline void adam_element(const AdamConsts& k, float factor, float g_in, float& m, float& v,
                         float& p) {
  const float g = factor * g_in;
  m = k.b1 * m + k.omb1 * g;
  v = k.b2 * v + k.omb2 * (g * g);
  p = p * k.decay;
  const float denom = std::sqrt(v) + k.eps_hat;
  p = p - k.alpha * (m / denom);
}

inline uint16_t bf16_round(float f) {
  uint32_t u;
  std::memcpy(&u, &f, 4);
  // reading: IEEE 754 fixes only that a NaN converts to a NaN, not which
  // one; this oracle returns the quiet NaN 0x7fc0, and parity compares bf16
  // NaNs by class (any NaN matches any NaN).
  if ((u & 0x7fffffffu) > 0x7f800000u) return 0x7fc0;
  u += 0x7fffu + ((u >> 16) & 1u);
  return (uint16_t)(u >> 16);
}

inline float bf16_value(uint16_t h) {
  uint32_t u = (uint32_t)h << 16;
  float f;
  std::memcpy(&f, &u, 4);
  return f;
}

// reading (quantiser): symmetric int8 for m with scale = max |m| of the
// block, unsigned uint8 for v with scale = max v of the block. Dequantised
// value = code * (scale / 127) (resp. / 255). Code = round-half-even of
// x * (127 / scale) (resp. 255 / scale), saturated to [-127, 127] (resp.
// [0, 255]), NaN giving 0; a zero scale means all codes 0. The m quantiser is
// symmetric: codes are clamped to [-127, 127], never -128, so no code
// dequantises above the block's absmax. The clamp matters when the scale is
// so small (subnormal) that 127 / scale overflows to infinity: every nonzero
// element then saturates, to +127 or -127 alike.
inline int8_t quant_m(float x, float inv) {
  const float y = x * inv;
  if (std::isnan(y)) return 0;
  return (int8_t)(int)std::nearbyint(std::fmin(std::fmax(y, -127.0f), 127.0f));
}
inline uint8_t quant_v(float x, float inv) {
  const float y = x * inv;
  if (std::isnan(y)) return 0;
  return (uint8_t)(int)std::nearbyint(std::fmin(std::fmax(y, 0.0f), 255.0f));
}

}  // namespace

extern "C" {

// ---------------------------------------------------------------- layout

// Shard atom and alignment of each tensor; returns 0 or -1 on a bad descriptor.
int orc_atoms(int n, const int64_t* rows, const int64_t* cols, const int32_t* gran,
              const int64_t* block_rows, const int64_t* tile_cols, int64_t g_coll,
              int64_t* block_out, int64_t* align_out) {
  std::vector<Tensor> ts;
  if (!make_tensors(n, rows, cols, gran, block_rows, tile_cols, g_coll, ts)) return -1;
  for (int t = 0; t < n; ++t) {
    block_out[t] = ts[t].block;
    align_out[t] = ts[t].align;
  }
  return 0;
}

// Plans the layout ([VSF] 核心方法 › Algorithm 1) for one order policy (or for
// an explicit permutation `order`, when it is non-null). Writes S and the
// per-tensor offsets into the m*S buffer. Returns 0, or -1 on bad input, or
// -2 if no S was found.
int orc_plan(int n, const int64_t* rows, const int64_t* cols, const int32_t* gran,
             const int64_t* block_rows, const int64_t* tile_cols, int64_t m, int64_t g_coll,
             int policy, const int32_t* order, int64_t* S_out, int64_t* offsets_out) {
  std::vector<Tensor> ts;
  if (m <= 0 || !make_tensors(n, rows, cols, gran, block_rows, tile_cols, g_coll, ts)) return -1;
  std::vector<int64_t> off;
  if (order != nullptr) {
    std::vector<int> ord(order, order + n);
    int64_t S = min_S_for_order(ts, ord, m, g_coll, off);
    if (S < 0) return -2;
    *S_out = S;
    std::copy(off.begin(), off.end(), offsets_out);
    return 0;
  }
  if (policy == ORDER_BEST3) {
    int64_t best = -1;
    std::vector<int64_t> best_off;
    for (int p : {ORDER_DEFAULT, ORDER_BLOCK, ORDER_SHAPE}) {
      int64_t S = min_S_for_order(ts, make_order(ts, p), m, g_coll, off);
      if (S >= 0 && (best < 0 || S < best)) {
        best = S;
        best_off = off;
      }
    }
    if (best < 0) return -2;
    *S_out = best;
    std::copy(best_off.begin(), best_off.end(), offsets_out);
    return 0;
  }
  if (policy < ORDER_DEFAULT || policy > ORDER_SHAPE) return -1;
  int64_t S = min_S_for_order(ts, make_order(ts, policy), m, g_coll, off);
  if (S < 0) return -2;
  *S_out = S;
  std::copy(off.begin(), off.end(), offsets_out);
  return 0;
}

// Brute force over every tensor order (n <= 9): the smallest S any order
// reaches with the same placement rule. Writes the first order reaching it.
int64_t orc_bruteforce_S(int n, const int64_t* rows, const int64_t* cols, const int32_t* gran,
                         const int64_t* block_rows, const int64_t* tile_cols, int64_t m,
                         int64_t g_coll, int32_t* best_order) {
  std::vector<Tensor> ts;
  if (n > 9 || m <= 0 || !make_tensors(n, rows, cols, gran, block_rows, tile_cols, g_coll, ts))
    return -1;
  std::vector<int> ord(n);
  std::iota(ord.begin(), ord.end(), 0);
  std::vector<int64_t> off;
  int64_t best = -1;
  do {
    int64_t S = min_S_for_order(ts, ord, m, g_coll, off);
    if (S >= 0 && (best < 0 || S < best)) {
      best = S;
      if (best_order) std::copy(ord.begin(), ord.end(), best_order);
    }
  } while (std::next_permutation(ord.begin(), ord.end()));
  return best;
}

// Exhaustive search on micro instances: the smallest S (a multiple of g_coll)
// for which SOME assignment of aligned, non-overlapping offsets, in any order,
// keeps every atom inside one rank ([VSF] Algorithm 1's constraints, without
// the heuristic). Exponential; meant for a few tensors and m*S of a few
// hundred elements. Returns -1 past `max_S`.
static bool exhaustive_fill(const std::vector<Tensor>& ts, int64_t m, int64_t S, int t,
                            std::vector<int64_t>& lo, std::vector<int64_t>& hi) {
  if (t == (int)ts.size()) return true;
  const Tensor& x = ts[t];
  for (int64_t o = 0; o + x.numel <= m * S; o += x.align) {
    bool ok = true;
    for (int64_t k = o / S + 1; k * S < o + x.numel; ++k)
      if ((k * S - o) % x.block != 0) ok = false;
    for (int u = 0; ok && u < t; ++u)
      if (o < hi[u] && lo[u] < o + x.numel) ok = false;
    if (!ok) continue;
    lo[t] = o;
    hi[t] = o + x.numel;
    if (exhaustive_fill(ts, m, S, t + 1, lo, hi)) return true;
  }
  return false;
}

int64_t orc_exhaustive_S(int n, const int64_t* rows, const int64_t* cols, const int32_t* gran,
                         const int64_t* block_rows, const int64_t* tile_cols, int64_t m,
                         int64_t g_coll, int64_t max_S) {
  std::vector<Tensor> ts;
  if (m <= 0 || !make_tensors(n, rows, cols, gran, block_rows, tile_cols, g_coll, ts)) return -1;
  std::vector<int64_t> lo(n), hi(n);
  for (int64_t S = lower_bound_S(ts, m, g_coll); S <= max_S; S += g_coll)
    if (exhaustive_fill(ts, m, S, 0, lo, hi)) return S;
  return -1;
}

// Quantisation blocks of the planned buffer, in tensor order ([VSF] 结构感知
// 训练 case study › 8-bit Adam; per-block scales). reading: ROWS tensors have
// one block per block_rows rows; TILE tensors one per block_rows x tile_cols
// tile, stripes top to bottom and tiles left to right; ELEM tensors one per
// g_coll consecutive elements from the tensor start. The last block of a
// tensor may be short. Each block is a row-major region: `base` (buffer
// element index of its first element), `nrows` rows of `ncols` elements,
// `stride` elements apart. With out arrays null, only counts the blocks.
int64_t orc_qblocks(int n, const int64_t* rows, const int64_t* cols, const int32_t* gran,
                    const int64_t* block_rows, const int64_t* tile_cols, int64_t g_coll,
                    const int64_t* offsets, int32_t* tensor_out, int64_t* base_out,
                    int64_t* nrows_out, int64_t* ncols_out, int64_t* stride_out) {
  std::vector<Tensor> ts;
  if (!make_tensors(n, rows, cols, gran, block_rows, tile_cols, g_coll, ts)) return -1;
  int64_t q = 0;
  auto emit = [&](int t, int64_t base, int64_t r, int64_t c, int64_t s) {
    if (tensor_out) {
      tensor_out[q] = t;
      base_out[q] = base;
      nrows_out[q] = r;
      ncols_out[q] = c;
      stride_out[q] = s;
    }
    ++q;
  };
  for (int t = 0; t < n; ++t) {
    const Tensor& x = ts[t];
    const int64_t off = offsets ? offsets[t] : 0;
    if (x.gran == GRAN_ELEM) {
      for (int64_t e = 0; e < x.numel; e += g_coll) {
        int64_t len = std::min(g_coll, x.numel - e);
        emit(t, off + e, 1, len, len);
      }
    } else if (x.gran == GRAN_ROWS) {
      for (int64_t r = 0; r < x.rows; r += x.block_rows) {
        int64_t nr = std::min(x.block_rows, x.rows - r);
        emit(t, off + r * x.cols, nr, x.cols, x.cols);
      }
    } else {
      for (int64_t r = 0; r < x.rows; r += x.block_rows) {
        int64_t nr = std::min(x.block_rows, x.rows - r);
        for (int64_t c = 0; c < x.cols; c += x.tile_cols) {
          int64_t nc = std::min(x.tile_cols, x.cols - c);
          emit(t, off + r * x.cols + c, nr, nc, x.cols);
        }
      }
    }
  }
  return q;
}

// ---------------------------------------------------------------- copy-in / copy-out

// Copy-in ([FSDP] 关键观察; [VSF] 核心方法 › Distributed Buffer, group copy):
// packed[offset_t + i] = tensor_t[i] for every real element. Element size 2
// (bf16 bits) or 4 (fp32). Padding is left as it is.
void orc_pack(int n, const void* const* tensors, const int64_t* numel, const int64_t* offsets,
              int esize, void* packed) {
  for (int t = 0; t < n; ++t) {
    const unsigned char* src = static_cast<const unsigned char*>(tensors[t]);
    unsigned char* dst = static_cast<unsigned char*>(packed) + offsets[t] * esize;
    for (int64_t i = 0; i < numel[t] * esize; ++i) dst[i] = src[i];
  }
}

// Copy-out: tensor_t[i] = packed[offset_t + i].
void orc_unpack(int n, void* const* tensors, const int64_t* numel, const int64_t* offsets,
                int esize, const void* packed) {
  for (int t = 0; t < n; ++t) {
    unsigned char* dst = static_cast<unsigned char*>(tensors[t]);
    const unsigned char* src = static_cast<const unsigned char*>(packed) + offsets[t] * esize;
    for (int64_t i = 0; i < numel[t] * esize; ++i) dst[i] = src[i];
  }
}

// ---------------------------------------------------------------- fused group ops

// One element-wise group op over every real element of a packed buffer, all
// tensors at once ([VSF] 核心方法 › Distributed Buffer: add / scale / zero
// applied across tensors). op 0: dst = 0; op 1: dst = dst * alpha; op 2:
// dst = dst + src. Arithmetic in fp32, one rounding, then to the buffer type
// (bf16 round-half-even for bf16 buffers). Padding is left as it is.
void orc_group_op(int op, int n, const int64_t* numel, const int64_t* offsets, void* dst,
                  int dst_bf16, const void* src, int src_bf16, float alpha) {
  for (int t = 0; t < n; ++t) {
    for (int64_t i = 0; i < numel[t]; ++i) {
      const int64_t e = offsets[t] + i;
      const float d = dst_bf16 ? bf16_value(static_cast<uint16_t*>(dst)[e])
                               : static_cast<float*>(dst)[e];
      float r = 0.0f;
      if (op == 1) r = d * alpha;
      if (op == 2) {
        const float x = src_bf16 ? bf16_value(static_cast<const uint16_t*>(src)[e])
                                 : static_cast<const float*>(src)[e];
        r = d + x;
      }
      if (dst_bf16)
        static_cast<uint16_t*>(dst)[e] = bf16_round(r);
      else
        static_cast<float*>(dst)[e] = r;
    }
  }
}

// ---------------------------------------------------------------- group norm and scale

// Sum of squares of every real gradient element, in fp64, tensors in order,
// elements in order ([VSF] 核心方法 › Distributed Buffer: fused group ops;
// the global norm behind gradient clipping). is_bf16: elements are bf16 bits.
double orc_sumsq(int n, const void* const* tensors, const int64_t* numel, int is_bf16) {
  double acc = 0.0;
  for (int t = 0; t < n; ++t) {
    for (int64_t i = 0; i < numel[t]; ++i) {
      double x = is_bf16 ? (double)bf16_value(static_cast<const uint16_t*>(tensors[t])[i])
                         : (double)static_cast<const float*>(tensors[t])[i];
      acc += x * x;
    }
  }
  return acc;
}

// Group scale factor applied to the summed gradient. reading: the packed
// gradient is the reduce-scatter SUM over `world` ranks, so the mean gradient
// is g/world and its norm sqrt(sumsq)/world; clipping scales by
// c = min(1, max_norm / (norm + 1e-6)) when max_norm is finite and positive
// (c = 1 otherwise); factor = fp32(c / world).
float orc_factor(double sumsq, int world, double max_norm, double* norm_out) {
  const double norm = std::sqrt(sumsq) / (double)world;
  double c = 1.0;
  if (std::isfinite(max_norm) && max_norm > 0.0) {
    double r = max_norm / (norm + 1e-6);
    if (r < 1.0) c = r;
  }
  if (norm_out) *norm_out = norm;
  return (float)(c / (double)world);
}

// ---------------------------------------------------------------- AdamW, one block

// One AdamW step on one quantisation block, elements given in the block's
// row-major order ([VSF] 结构感知训练 case study › 8-bit Adam: the block is
// local to one rank, so its scale needs no exchange).
//   g_in:  gradient (bf16 bits if grad_bf16, else fp32)
//   quantized != 0: mq (int8 codes) / vq (uint8 codes) and *m_scale / *v_scale
//       hold the state; they are overwritten with the requantised state.
//       reading: the update uses the fresh fp32 m and v; requantisation
//       follows, with the new block scales.
//   quantized == 0: m32 / v32 hold the fp32 state and are updated in place.
//   p: fp32 master, updated in place; bf16_out: RNE copy of the new master.
void orc_adam_block(int64_t count, const void* g_in, int grad_bf16, float factor, int quantized,
                    int8_t* mq, uint8_t* vq, float* m_scale, float* v_scale, float* m32,
                    float* v32, float* p, uint16_t* bf16_out, double lr, double beta1,
                    double beta2, double eps, double wd, int step) {
  std::fesetround(FE_TONEAREST);
  const AdamConsts k = adam_consts(lr, beta1, beta2, eps, wd, step);
  std::vector<float> M(count), V(count);
  float dm = 0.0f, dv = 0.0f;
  if (quantized) {
    dm = *m_scale / 127.0f;
    dv = *v_scale / 255.0f;
  }
  for (int64_t i = 0; i < count; ++i) {
    const float g = grad_bf16 ? bf16_value(static_cast<const uint16_t*>(g_in)[i])
                              : static_cast<const float*>(g_in)[i];
    float m = quantized ? (float)mq[i] * dm : m32[i];
    float v = quantized ? (float)vq[i] * dv : v32[i];
    adam_element(k, factor, g, m, v, p[i]);
    M[i] = m;
    V[i] = v;
    bf16_out[i] = bf16_round(p[i]);
  }
  if (!quantized) {
    for (int64_t i = 0; i < count; ++i) {
      m32[i] = M[i];
      v32[i] = V[i];
    }
    return;
  }
  float sm = 0.0f, sv = 0.0f;
  for (int64_t i = 0; i < count; ++i) {
    sm = std::fmax(sm, std::fabs(M[i]));
    sv = std::fmax(sv, V[i]);
  }
  const float im = sm > 0.0f ? 127.0f / sm : 0.0f;
  const float iv = sv > 0.0f ? 255.0f / sv : 0.0f;
  for (int64_t i = 0; i < count; ++i) {
    mq[i] = sm > 0.0f ? quant_m(M[i], im) : (int8_t)0;
    vq[i] = sv > 0.0f ? quant_v(V[i], iv) : (uint8_t)0;
  }
  *m_scale = sm;
  *v_scale = sv;
}

// The same step over every block of a packed buffer: gathers each block's
// elements (row-major), runs orc_adam_block, scatters the results back.
// Buffers are the m*S packed arrays; in fp32-state mode m_state/v_state are
// float arrays, otherwise int8/uint8 code arrays.
void orc_adam_all(int64_t nblocks, const int64_t* base, const int64_t* nrows,
                  const int64_t* ncols, const int64_t* stride, const void* packed_grad,
                  int grad_bf16, float factor, int quantized, void* m_state, void* v_state,
                  float* m_scale, float* v_scale, float* master, uint16_t* packed_bf16,
                  double lr, double beta1, double beta2, double eps, double wd, int step) {
  const int gsz = grad_bf16 ? 2 : 4;
  for (int64_t q = 0; q < nblocks; ++q) {
    const int64_t cnt = nrows[q] * ncols[q];
    std::vector<unsigned char> g(cnt * gsz);
    std::vector<int8_t> mq(cnt);
    std::vector<uint8_t> vq(cnt);
    std::vector<float> m32(cnt), v32(cnt), p(cnt);
    std::vector<uint16_t> bf(cnt);
    for (int64_t r = 0, i = 0; r < nrows[q]; ++r) {
      for (int64_t c = 0; c < ncols[q]; ++c, ++i) {
        const int64_t e = base[q] + r * stride[q] + c;
        std::memcpy(&g[i * gsz], static_cast<const unsigned char*>(packed_grad) + e * gsz, gsz);
        if (quantized) {
          mq[i] = static_cast<int8_t*>(m_state)[e];
          vq[i] = static_cast<uint8_t*>(v_state)[e];
        } else {
          m32[i] = static_cast<float*>(m_state)[e];
          v32[i] = static_cast<float*>(v_state)[e];
        }
        p[i] = master[e];
      }
    }
    orc_adam_block(cnt, g.data(), grad_bf16, factor, quantized, mq.data(), vq.data(),
                   quantized ? &m_scale[q] : nullptr, quantized ? &v_scale[q] : nullptr,
                   m32.data(), v32.data(), p.data(), bf.data(), lr, beta1, beta2, eps, wd, step);
    for (int64_t r = 0, i = 0; r < nrows[q]; ++r) {
      for (int64_t c = 0; c < ncols[q]; ++c, ++i) {
        const int64_t e = base[q] + r * stride[q] + c;
        if (quantized) {
          static_cast<int8_t*>(m_state)[e] = mq[i];
          static_cast<uint8_t*>(v_state)[e] = vq[i];
        } else {
          static_cast<float*>(m_state)[e] = m32[i];
          static_cast<float*>(v_state)[e] = v32[i];
        }
        master[e] = p[i];
        packed_bf16[e] = bf[i];
      }
    }
  }
}

// Quantiser on its own (for its property tests): codes and scale of one
// block of fp32 values, and the dequantised values.
void orc_quantize_m(int64_t count, const float* x, int8_t* codes, float* scale, float* deq) {
  std::fesetround(FE_TONEAREST);
  float s = 0.0f;
  for (int64_t i = 0; i < count; ++i) s = std::fmax(s, std::fabs(x[i]));
  const float inv = s > 0.0f ? 127.0f / s : 0.0f;
  for (int64_t i = 0; i < count; ++i) codes[i] = s > 0.0f ? quant_m(x[i], inv) : (int8_t)0;
  *scale = s;
  const float d = s / 127.0f;
  for (int64_t i = 0; i < count; ++i) deq[i] = (float)codes[i] * d;
}

void orc_quantize_v(int64_t count, const float* x, uint8_t* codes, float* scale, float* deq) {
  std::fesetround(FE_TONEAREST);
  float s = 0.0f;
  for (int64_t i = 0; i < count; ++i) s = std::fmax(s, x[i]);
  const float inv = s > 0.0f ? 255.0f / s : 0.0f;
  for (int64_t i = 0; i < count; ++i) codes[i] = s > 0.0f ? quant_v(x[i], inv) : (uint8_t)0;
  *scale = s;
  const float d = s / 255.0f;
  for (int64_t i = 0; i < count; ++i) deq[i] = (float)codes[i] * d;
}

uint16_t orc_bf16_round(float f) { return bf16_round(f); }

}  // extern "C"
