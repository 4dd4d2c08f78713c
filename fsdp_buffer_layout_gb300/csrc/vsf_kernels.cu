// vsf_kernels.cu — sm_103a kernels and the per-step C ABI of libvsf.
//
// Per step, on the caller's stream (all device memory caller-owned):
//   vsf_pack              copy-in of every gradient tensor into the planned
//                         m*S buffer, fused with the sum of squares
//                         ("FSDP" concept page › 关键观察: copy cost;
//                         "veScale-FSDP: Flexible and High-Performance FSDP at
//                         Scale (MLSys 2026)" summary page › 核心方法 ›
//                         Distributed Buffer: fused group copy / scale);
//   vsf_group_norm_scale  one CTA turns the partial sums into the clip and
//                         1/world factor;
//   vsf_adam8_step        block-wise 8-bit AdamW on every rank's RaggedShard
//                         slice (same page › 结构感知训练 case study › 8-bit
//                         Adam): one HBM pass per block, the block's new
//                         absmax reduced across a thread-block cluster;
//   vsf_unpack            copy-out of the bf16 parameters.
// Nothing here is a dense contraction: the kernels are HBM-bound streams
// (128-bit loads and stores, streaming cache hints, warp-shuffle reductions).
//
// Floating point: every fp32 operation of the AdamW update, the quantiser and
// the squared-norm accumulation is written with an explicit round-to-nearest
// intrinsic (__fmul_rn, __fadd_rn, __fdiv_rn, __fsqrt_rn, ...), which the
// compiler never contracts into an FMA, so each operation rounds once in the
// order written.
#include <cooperative_groups.h>
#include <cuda_runtime.h>

#include <cmath>
#include <cstring>
#include <string>

#include "vsf_internal.h"

namespace cg = cooperative_groups;

namespace vsf {
namespace {

constexpr int kCopyThreads = 256;
constexpr int kCopyCtasPerSm = 8;
constexpr int kAdamThreads = 512;
constexpr int kMaxCluster = 8;
constexpr int kSmallThreads = 256;

struct TensorPtrs {
  const void* p[kMaxTensors];
};

struct AdamConsts {
  float b1, omb1, b2, omb2, eps, decay, step_size, bc2s;
};

// ------------------------------------------------------------------ helpers

__device__ __forceinline__ float bf16_to_f32(uint32_t h) { return __uint_as_float(h << 16); }

__device__ __forceinline__ uint32_t f32_to_bf16(float f) {
  uint32_t u = __float_as_uint(f);
  if ((u & 0x7fffffffu) > 0x7f800000u) return 0x7fc0u;  // NaN -> canonical quiet NaN
  u += 0x7fffu + ((u >> 16) & 1u);
  return u >> 16;
}

// Double-float accumulator of non-negative terms (Knuth's TwoSum keeps the
// rounding error of every addition).
struct DF {
  float hi = 0.0f, lo = 0.0f;
  __device__ __forceinline__ void add(float x) {
    const float s = __fadd_rn(hi, x);
    const float bp = __fsub_rn(s, hi);
    const float err = __fadd_rn(__fsub_rn(hi, __fsub_rn(s, bp)), __fsub_rn(x, bp));
    hi = s;
    lo = __fadd_rn(lo, err);
  }
};

// x*x into the accumulator, exactly for bf16 inputs (16 significant bits)
// and with the FMA-recovered product error for fp32 inputs.
__device__ __forceinline__ void acc_sq(DF& a, float x) {
  const float p = __fmul_rn(x, x);
  a.add(p);
  a.lo = __fadd_rn(a.lo, __fmaf_rn(x, x, -p));
}

__device__ __forceinline__ int64_t min64(int64_t a, int64_t b) { return a < b ? a : b; }

__device__ __forceinline__ float warp_max(float x) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) x = fmaxf(x, __shfl_xor_sync(0xffffffffu, x, o));
  return x;
}

__device__ __forceinline__ double warp_sum(double x) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
  return x;
}

// Streaming (evict-first) 128-bit accesses for data touched once.
__device__ __forceinline__ uint4 ld_stream(const void* p) { return __ldcs(reinterpret_cast<const uint4*>(p)); }
__device__ __forceinline__ void st_stream(void* p, uint4 v) { __stcs(reinterpret_cast<uint4*>(p), v); }

// ------------------------------------------------------------------ copy-in / copy-out

enum CopyMode { kPack = 0, kUnpack = 1, kNormOnly = 2 };

template <typename T>
__device__ __forceinline__ void sq_vec(DF& acc, uint4 v);

template <>
__device__ __forceinline__ void sq_vec<uint16_t>(DF& acc, uint4 v) {
  const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    acc_sq(acc, bf16_to_f32(w[i] & 0xffffu));
    acc_sq(acc, bf16_to_f32(w[i] >> 16));
  }
}

template <>
__device__ __forceinline__ void sq_vec<float>(DF& acc, uint4 v) {
  acc_sq(acc, __uint_as_float(v.x));
  acc_sq(acc, __uint_as_float(v.y));
  acc_sq(acc, __uint_as_float(v.z));
  acc_sq(acc, __uint_as_float(v.w));
}

__device__ __forceinline__ float elem_f32(uint16_t h) { return bf16_to_f32(h); }
__device__ __forceinline__ float elem_f32(float f) { return f; }

// One CTA copies its span of the concatenated real elements (tensor order).
// kPack:     packed[off_t + i] = tensor_t[i], and sum of squares.
// kUnpack:   tensor_t[i] = packed[off_t + i].
// kNormOnly: sum of squares of packed[off_t + i].
template <typename T, int kMode>
__global__ void __launch_bounds__(kCopyThreads) copy_kernel(TensorPtrs ptrs,
                                                            const int64_t* __restrict__ t_off,
                                                            const int64_t* __restrict__ t_numel,
                                                            const CopySpan* __restrict__ spans,
                                                            T* packed, double* partials) {
  constexpr int V = 16 / sizeof(T);
  const CopySpan s0 = spans[blockIdx.x];
  const CopySpan s1 = spans[blockIdx.x + 1];
  DF acc;
  for (int t = s0.tensor; t <= s1.tensor; ++t) {
    const int64_t b = (t == s0.tensor) ? s0.elem : 0;
    const int64_t e = (t == s1.tensor) ? s1.elem : t_numel[t];
    if (b >= e) continue;
    T* pk = packed + t_off[t];
    T* tp = const_cast<T*>(static_cast<const T*>(ptrs.p[t]));
    const T* src = (kMode == kUnpack) ? pk : (kMode == kPack ? tp : pk);
    T* dst = (kMode == kUnpack) ? tp : pk;
    const bool aligned = ((reinterpret_cast<uintptr_t>(src + b) |
                           (kMode == kNormOnly ? 0 : reinterpret_cast<uintptr_t>(dst + b))) &
                          15) == 0;
    int64_t i = b;
    if (aligned) {
      const int64_t nvec = (e - b) / V;
      const uint4* s = reinterpret_cast<const uint4*>(src + b);
      uint4* d = reinterpret_cast<uint4*>(dst + b);
      int64_t k = threadIdx.x;
      for (; k + 3 * kCopyThreads < nvec; k += 4 * kCopyThreads) {
        uint4 r[4];
#pragma unroll
        for (int u = 0; u < 4; ++u) r[u] = ld_stream(s + k + u * kCopyThreads);
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          if (kMode != kUnpack) sq_vec<T>(acc, r[u]);
          if (kMode != kNormOnly) st_stream(d + k + u * kCopyThreads, r[u]);
        }
      }
      for (; k < nvec; k += kCopyThreads) {
        const uint4 r = ld_stream(s + k);
        if (kMode != kUnpack) sq_vec<T>(acc, r);
        if (kMode != kNormOnly) st_stream(d + k, r);
      }
      i = b + nvec * V;
    }
    for (int64_t j = i + threadIdx.x; j < e; j += kCopyThreads) {
      const T x = src[j];
      if (kMode != kUnpack) acc_sq(acc, elem_f32(x));
      if (kMode != kNormOnly) dst[j] = x;
    }
  }
  if (kMode == kUnpack) return;
  __shared__ double red[kCopyThreads / 32];
  double v = warp_sum((double)acc.hi + (double)acc.lo);
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = v;
  __syncthreads();
  if (threadIdx.x == 0) {
    double s = 0.0;
    for (int w = 0; w < kCopyThreads / 32; ++w) s += red[w];
    partials[blockIdx.x] = s;
  }
}

// One CTA: fixed-order fp64 sum of the per-CTA partials, then the group
// scale factor (clip and 1/world).
__global__ void __launch_bounds__(256) norm_finalize_kernel(const double* __restrict__ partials,
                                                            int n, int world, double max_norm,
                                                            float* d_factor, double* d_norm) {
  __shared__ double red[256];
  double s = 0.0;
  for (int i = threadIdx.x; i < n; i += 256) s += partials[i];
  red[threadIdx.x] = s;
  __syncthreads();
  for (int w = 128; w > 0; w >>= 1) {
    if (threadIdx.x < w) red[threadIdx.x] += red[threadIdx.x + w];
    __syncthreads();
  }
  if (threadIdx.x == 0) {
    const double norm = sqrt(red[0]) / (double)world;
    double c = 1.0;
    if (isfinite(max_norm) && max_norm > 0.0) {
      const double r = max_norm / (norm + 1e-6);
      if (r < 1.0) c = r;
    }
    *d_factor = __double2float_rn(c / (double)world);
    if (d_norm) *d_norm = norm;
  }
}

// ------------------------------------------------------------------ AdamW

__device__ __forceinline__ void moments(const AdamConsts& k, float factor, float gin, float dm,
                                        float dv, int qm, int qv, float& m, float& v) {
  const float g = __fmul_rn(factor, gin);
  const float mp = __fmul_rn(__int2float_rn(qm), dm);
  const float vp = __fmul_rn(__int2float_rn(qv), dv);
  m = __fadd_rn(__fmul_rn(k.b1, mp), __fmul_rn(k.omb1, g));
  v = __fadd_rn(__fmul_rn(k.b2, vp), __fmul_rn(k.omb2, __fmul_rn(g, g)));
}

__device__ __forceinline__ float update_master(const AdamConsts& k, float p, float m, float v) {
  p = __fmul_rn(p, k.decay);
  const float denom = __fadd_rn(__fdiv_rn(__fsqrt_rn(v), k.bc2s), k.eps);
  return __fsub_rn(p, __fmul_rn(k.step_size, __fdiv_rn(m, denom)));
}

__device__ __forceinline__ int quant_m(float m, float inv, bool on) {
  if (!on) return 0;
  return __float2int_rn(fminf(fmaxf(__fmul_rn(m, inv), -127.0f), 127.0f));
}
__device__ __forceinline__ int quant_v(float v, float inv, bool on) {
  if (!on) return 0;
  return __float2int_rn(fminf(fmaxf(__fmul_rn(v, inv), 0.0f), 255.0f));
}

// Inputs of up to 8 consecutive elements: gradient, m code, v code.
template <typename GT>
struct Group {
  float g[8];
  int qm[8], qv[8];
};

template <typename GT>
__device__ __forceinline__ void load_group(const GT* grad, const int8_t* mq, const uint8_t* vq,
                                           int64_t e, int cnt, bool vec, Group<GT>& G) {
  if (vec && cnt == 8) {
    if constexpr (sizeof(GT) == 2) {
      const uint4 r = __ldg(reinterpret_cast<const uint4*>(grad + e));
      const uint32_t w[4] = {r.x, r.y, r.z, r.w};
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        G.g[2 * i] = bf16_to_f32(w[i] & 0xffffu);
        G.g[2 * i + 1] = bf16_to_f32(w[i] >> 16);
      }
    } else {
      const float4 a = __ldg(reinterpret_cast<const float4*>(grad + e));
      const float4 b = __ldg(reinterpret_cast<const float4*>(grad + e) + 1);
      G.g[0] = a.x; G.g[1] = a.y; G.g[2] = a.z; G.g[3] = a.w;
      G.g[4] = b.x; G.g[5] = b.y; G.g[6] = b.z; G.g[7] = b.w;
    }
    const uint2 cm = __ldg(reinterpret_cast<const uint2*>(mq + e));
    const uint2 cv = __ldg(reinterpret_cast<const uint2*>(vq + e));
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      G.qm[i] = (int)(int8_t)((cm.x >> (8 * i)) & 0xff);
      G.qm[4 + i] = (int)(int8_t)((cm.y >> (8 * i)) & 0xff);
      G.qv[i] = (int)((cv.x >> (8 * i)) & 0xff);
      G.qv[4 + i] = (int)((cv.y >> (8 * i)) & 0xff);
    }
  } else {
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      if (i < cnt) {
        G.g[i] = elem_f32(grad[e + i]);
        G.qm[i] = mq[e + i];
        G.qv[i] = vq[e + i];
      } else {
        G.g[i] = 0.0f;
        G.qm[i] = 0;
        G.qv[i] = 0;
      }
    }
  }
}

struct BlockCtx {
  float dm, dv;        // old scales / 127, / 255
  float im, iv;        // 127 / new m scale, 255 / new v scale
  bool mon, von;       // new scales non-zero
};

// Phase 1 on one group: the new moments' maxima.
template <typename GT>
__device__ __forceinline__ void group_phase1(const AdamConsts& k, float factor, const BlockCtx& c,
                                             const GT* grad, const int8_t* mq, const uint8_t* vq,
                                             int64_t e, int cnt, bool vec, float& mx, float& vx) {
  Group<GT> G;
  load_group(grad, mq, vq, e, cnt, vec, G);
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    if (i < cnt) {
      float m, v;
      moments(k, factor, G.g[i], c.dm, c.dv, G.qm[i], G.qv[i], m, v);
      mx = fmaxf(mx, fabsf(m));
      vx = fmaxf(vx, v);
    }
  }
}

// Phase 2 on one group: recompute the moments (bit-identical), update the
// master, requantise with the new scales, write everything.
template <typename GT>
__device__ __forceinline__ void group_phase2(const AdamConsts& k, float factor, const BlockCtx& c,
                                             const GT* grad, int8_t* mq, uint8_t* vq,
                                             float* master, uint16_t* bf, int64_t e, int cnt,
                                             bool vec) {
  Group<GT> G;
  load_group(grad, mq, vq, e, cnt, vec, G);
  float p[8];
  if (vec && cnt == 8) {
    const float4 a = __ldcs(reinterpret_cast<const float4*>(master + e));
    const float4 b = __ldcs(reinterpret_cast<const float4*>(master + e) + 1);
    p[0] = a.x; p[1] = a.y; p[2] = a.z; p[3] = a.w;
    p[4] = b.x; p[5] = b.y; p[6] = b.z; p[7] = b.w;
  } else {
#pragma unroll
    for (int i = 0; i < 8; ++i) p[i] = i < cnt ? master[e + i] : 0.0f;
  }
  uint32_t cm[2] = {0, 0}, cv[2] = {0, 0}, hb[4] = {0, 0, 0, 0};
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    float m, v;
    moments(k, factor, G.g[i], c.dm, c.dv, G.qm[i], G.qv[i], m, v);
    p[i] = update_master(k, p[i], m, v);
    const uint32_t qm = (uint32_t)(quant_m(m, c.im, c.mon) & 0xff);
    const uint32_t qv = (uint32_t)quant_v(v, c.iv, c.von);
    cm[i >> 2] |= qm << (8 * (i & 3));
    cv[i >> 2] |= qv << (8 * (i & 3));
    hb[i >> 1] |= f32_to_bf16(p[i]) << (16 * (i & 1));
  }
  if (vec && cnt == 8) {
    __stcs(reinterpret_cast<float4*>(master + e), make_float4(p[0], p[1], p[2], p[3]));
    __stcs(reinterpret_cast<float4*>(master + e) + 1, make_float4(p[4], p[5], p[6], p[7]));
    st_stream(bf + e, make_uint4(hb[0], hb[1], hb[2], hb[3]));
    __stcs(reinterpret_cast<uint2*>(mq + e), make_uint2(cm[0], cm[1]));
    __stcs(reinterpret_cast<uint2*>(vq + e), make_uint2(cv[0], cv[1]));
  } else {
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      if (i < cnt) {
        master[e + i] = p[i];
        bf[e + i] = (uint16_t)((hb[i >> 1] >> (16 * (i & 1))) & 0xffffu);
        mq[e + i] = (int8_t)((cm[i >> 2] >> (8 * (i & 3))) & 0xff);
        vq[e + i] = (uint8_t)((cv[i >> 2] >> (8 * (i & 3))) & 0xff);
      }
    }
  }
}

// Row / tile blocks: one thread-block cluster per quantisation block. Each
// CTA of the cluster takes an equal share of the block; phase 1 reads the
// gradient and the codes (4 B per element for bf16 gradients) and reduces the
// new absmax; the CTAs exchange their maxima through distributed shared
// memory and one cluster barrier; phase 2 re-reads the same share (from L2:
// at most clusters x block bytes are in flight) plus the master and writes
// master, bf16 copy and codes. HBM sees each byte once.
template <typename GT>
__global__ void __launch_bounds__(kAdamThreads) adam_big_kernel(
    const QBlock* __restrict__ qb, const int32_t* __restrict__ list, int nlist, int nclusters,
    const GT* __restrict__ grad, const float* __restrict__ d_factor, float* master, int8_t* mq,
    uint8_t* vq, float* m_scale, float* v_scale, uint16_t* bf, AdamConsts k) {
  cg::cluster_group cluster = cg::this_cluster();
  const int CL = (int)cluster.num_blocks();
  const int crank = (int)cluster.block_rank();
  const int cid = blockIdx.x / CL;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  constexpr int kWarps = kAdamThreads / 32;
  __shared__ float red[2][2][kWarps];
  __shared__ float2 slots[2][kMaxCluster];
  const float factor = *d_factor;

  int par = 0;
  for (int j = cid; j < nlist; j += nclusters, par ^= 1) {
    const int q = list[j];
    const QBlock b = qb[q];
    BlockCtx c;
    c.dm = __fdiv_rn(m_scale[q], 127.0f);
    c.dv = __fdiv_rn(v_scale[q], 255.0f);
    const bool contiguous = b.nrows == 1;
    const bool vec = (b.base % 8 == 0) && (contiguous || b.stride % 8 == 0);

    // This CTA's share: vectors [v0, v1) of a contiguous block, or rows
    // [r0, r1) of a tiled block.
    int64_t v0 = 0, v1 = 0;
    int r0 = 0, r1 = 0;
    const int vpr = (b.ncols + 7) / 8;
    if (contiguous) {
      const int64_t nv = vpr;
      const int64_t per = (nv + CL - 1) / CL;
      v0 = min64(nv, (int64_t)crank * per);
      v1 = min64(nv, v0 + per);
    } else {
      const int per = (b.nrows + CL - 1) / CL;
      r0 = min(b.nrows, crank * per);
      r1 = min(b.nrows, r0 + per);
    }

    // phase 1
    float mx = 0.0f, vx = 0.0f;
    if (contiguous) {
      for (int64_t v = v0 + tid; v < v1; v += kAdamThreads) {
        const int64_t off = v * 8;
        group_phase1<GT>(k, factor, c, grad, mq, vq, b.base + off,
                         (int)min64(8, b.ncols - off), vec, mx, vx);
      }
    } else {
      for (int r = r0 + warp; r < r1; r += kWarps)
        for (int v = lane; v < vpr; v += 32)
          group_phase1<GT>(k, factor, c, grad, mq, vq, b.base + (int64_t)r * b.stride + v * 8,
                           min(8, b.ncols - v * 8), vec, mx, vx);
    }
    mx = warp_max(mx);
    vx = warp_max(vx);
    if (lane == 0) {
      red[par][0][warp] = mx;
      red[par][1][warp] = vx;
    }
    __syncthreads();
    if (tid == 0) {
      float bm = 0.0f, bv = 0.0f;
      for (int w = 0; w < kWarps; ++w) {
        bm = fmaxf(bm, red[par][0][w]);
        bv = fmaxf(bv, red[par][1][w]);
      }
      for (int r = 0; r < CL; ++r) *cluster.map_shared_rank(&slots[par][crank], r) = make_float2(bm, bv);
    }
    cluster.sync();
    float sm = 0.0f, sv = 0.0f;
    for (int r = 0; r < CL; ++r) {
      sm = fmaxf(sm, slots[par][r].x);
      sv = fmaxf(sv, slots[par][r].y);
    }
    c.mon = sm > 0.0f;
    c.von = sv > 0.0f;
    c.im = c.mon ? __fdiv_rn(127.0f, sm) : 0.0f;
    c.iv = c.von ? __fdiv_rn(255.0f, sv) : 0.0f;
    if (crank == 0 && tid == 0) {
      m_scale[q] = sm;
      v_scale[q] = sv;
    }

    // phase 2
    if (contiguous) {
      for (int64_t v = v0 + tid; v < v1; v += kAdamThreads) {
        const int64_t off = v * 8;
        group_phase2<GT>(k, factor, c, grad, mq, vq, master, bf, b.base + off,
                         (int)min64(8, b.ncols - off), vec);
      }
    } else {
      for (int r = r0 + warp; r < r1; r += kWarps)
        for (int v = lane; v < vpr; v += 32)
          group_phase2<GT>(k, factor, c, grad, mq, vq, master, bf,
                           b.base + (int64_t)r * b.stride + v * 8, min(8, b.ncols - v * 8), vec);
    }
  }
  cluster.sync();  // no CTA leaves while a peer may still write its slots
}

// Element-granular chunks (g_coll elements each): one warp per block, two
// passes over the (L1-resident) chunk.
template <typename GT>
__global__ void __launch_bounds__(kSmallThreads) adam_small_kernel(
    const QBlock* __restrict__ qb, const int32_t* __restrict__ list, int nlist,
    const GT* __restrict__ grad, const float* __restrict__ d_factor, float* master, int8_t* mq,
    uint8_t* vq, float* m_scale, float* v_scale, uint16_t* bf, AdamConsts k) {
  const int lane = threadIdx.x & 31;
  const int j = blockIdx.x * (kSmallThreads / 32) + (threadIdx.x >> 5);
  if (j >= nlist) return;
  const int q = list[j];
  const QBlock b = qb[q];
  const float factor = *d_factor;
  BlockCtx c;
  c.dm = __fdiv_rn(m_scale[q], 127.0f);
  c.dv = __fdiv_rn(v_scale[q], 255.0f);
  float mx = 0.0f, vx = 0.0f;
  for (int i = lane; i < b.ncols; i += 32) {
    float m, v;
    moments(k, factor, elem_f32(grad[b.base + i]), c.dm, c.dv, mq[b.base + i], vq[b.base + i],
            m, v);
    mx = fmaxf(mx, fabsf(m));
    vx = fmaxf(vx, v);
  }
  const float sm = warp_max(mx), sv = warp_max(vx);
  c.mon = sm > 0.0f;
  c.von = sv > 0.0f;
  c.im = c.mon ? __fdiv_rn(127.0f, sm) : 0.0f;
  c.iv = c.von ? __fdiv_rn(255.0f, sv) : 0.0f;
  for (int i = lane; i < b.ncols; i += 32) {
    const int64_t e = b.base + i;
    float m, v;
    moments(k, factor, elem_f32(grad[e]), c.dm, c.dv, mq[e], vq[e], m, v);
    const float p = update_master(k, master[e], m, v);
    master[e] = p;
    bf[e] = (uint16_t)f32_to_bf16(p);
    mq[e] = (int8_t)quant_m(m, c.im, c.mon);
    vq[e] = (uint8_t)quant_v(v, c.iv, c.von);
  }
  __syncwarp();
  if (lane == 0) {
    m_scale[q] = sm;
    v_scale[q] = sv;
  }
}

// fp32 moments (no quantisation): element-wise over the copy spans.
template <typename GT>
__global__ void __launch_bounds__(kCopyThreads) adam_fp32_kernel(
    const int64_t* __restrict__ t_off, const int64_t* __restrict__ t_numel,
    const CopySpan* __restrict__ spans, const GT* __restrict__ grad,
    const float* __restrict__ d_factor, float* master, float* m_state, float* v_state,
    uint16_t* bf, AdamConsts k) {
  const CopySpan s0 = spans[blockIdx.x];
  const CopySpan s1 = spans[blockIdx.x + 1];
  const float factor = *d_factor;
  for (int t = s0.tensor; t <= s1.tensor; ++t) {
    const int64_t b = (t == s0.tensor) ? s0.elem : 0;
    const int64_t e = (t == s1.tensor) ? s1.elem : t_numel[t];
    const int64_t base = t_off[t];
    for (int64_t i = b + threadIdx.x; i < e; i += kCopyThreads) {
      const int64_t x = base + i;
      const float g = __fmul_rn(factor, elem_f32(grad[x]));
      const float m = __fadd_rn(__fmul_rn(k.b1, m_state[x]), __fmul_rn(k.omb1, g));
      const float v = __fadd_rn(__fmul_rn(k.b2, v_state[x]), __fmul_rn(k.omb2, __fmul_rn(g, g)));
      const float p = update_master(k, master[x], m, v);
      m_state[x] = m;
      v_state[x] = v;
      master[x] = p;
      bf[x] = (uint16_t)f32_to_bf16(p);
    }
  }
}

// ------------------------------------------------------------------ host side

vsf_status cuda_fail(cudaError_t e, const char* what) {
  return fail(VSF_ERR_CUDA, std::string(what) + ": " + cudaGetErrorString(e));
}

bool misaligned(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15) != 0; }

vsf_status check_ready(const vsf_plan* plan, const char* who) {
  if (plan == nullptr) return fail(VSF_ERR_ARG, std::string(who) + ": NULL plan");
  if (!plan->uploaded)
    return fail(VSF_ERR_STATE, std::string(who) + ": plan not uploaded (call vsf_plan_upload)");
  int dev = -1;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(e, who);
  if (dev != plan->device)
    return fail(VSF_ERR_STATE, std::string(who) + ": current device differs from upload device");
  return VSF_OK;
}

template <typename T>
const T* ws_ptr(const vsf_plan* plan, size_t off) {
  return reinterpret_cast<const T*>(plan->d_ws + off);
}

AdamConsts make_consts(const vsf_adam_hparams& hp, int step) {
  double p1 = 1.0, p2 = 1.0;
  for (int i = 0; i < step; ++i) {
    p1 *= hp.beta1;
    p2 *= hp.beta2;
  }
  AdamConsts k;
  k.b1 = (float)hp.beta1;
  k.omb1 = (float)(1.0 - hp.beta1);
  k.b2 = (float)hp.beta2;
  k.omb2 = (float)(1.0 - hp.beta2);
  k.eps = (float)hp.eps;
  k.decay = (float)(1.0 - hp.lr * hp.weight_decay);
  k.step_size = (float)(hp.lr / (1.0 - p1));
  k.bc2s = (float)std::sqrt(1.0 - p2);
  return k;
}

template <typename T, int kMode>
vsf_status launch_copy(const vsf_plan* plan, const void* const* tensors, void* packed,
                       cudaStream_t st, const char* who) {
  TensorPtrs ptrs;
  std::memset(&ptrs, 0, sizeof(ptrs));
  if (kMode != kNormOnly) {
    if (plan->n > kMaxTensors)
      return fail(VSF_ERR_ARG, std::string(who) + ": more than 2048 tensors per call");
    if (tensors == nullptr) return fail(VSF_ERR_ARG, std::string(who) + ": NULL tensor array");
    for (int t = 0; t < plan->n; ++t) {
      if (tensors[t] == nullptr) return fail(VSF_ERR_ARG, std::string(who) + ": NULL tensor");
      if (misaligned(tensors[t]))
        return fail(VSF_ERR_ALIGN, std::string(who) + ": tensor " + std::to_string(t) +
                                       " not 16-byte aligned");
      ptrs.p[t] = tensors[t];
    }
  }
  copy_kernel<T, kMode><<<plan->copy_grid, kCopyThreads, 0, st>>>(
      ptrs, ws_ptr<int64_t>(plan, plan->layout.tensor_off),
      ws_ptr<int64_t>(plan, plan->layout.tensor_numel),
      ws_ptr<CopySpan>(plan, plan->layout.spans), static_cast<T*>(packed),
      reinterpret_cast<double*>(plan->d_ws + plan->layout.partials));
  cudaError_t e = cudaGetLastError();
  return e == cudaSuccess ? VSF_OK : cuda_fail(e, who);
}

template <typename GT>
vsf_status launch_adam(const vsf_plan* plan, const void* grad, const float* d_factor,
                       float* master, void* m_state, void* v_state, float* m_scale,
                       float* v_scale, uint16_t* bf, const AdamConsts& k, bool quantized,
                       cudaStream_t st) {
  const GT* g = static_cast<const GT*>(grad);
  const QBlock* qb = ws_ptr<QBlock>(plan, plan->layout.qblocks);
  if (!quantized) {
    adam_fp32_kernel<GT><<<plan->copy_grid, kCopyThreads, 0, st>>>(
        ws_ptr<int64_t>(plan, plan->layout.tensor_off),
        ws_ptr<int64_t>(plan, plan->layout.tensor_numel),
        ws_ptr<CopySpan>(plan, plan->layout.spans), g, d_factor, master,
        static_cast<float*>(m_state), static_cast<float*>(v_state), bf, k);
    cudaError_t e = cudaGetLastError();
    return e == cudaSuccess ? VSF_OK : cuda_fail(e, "vsf_adam8_step");
  }
  int8_t* mq = static_cast<int8_t*>(m_state);
  uint8_t* vq = static_cast<uint8_t*>(v_state);
  const int nbig = (int)plan->big_blocks.size();
  if (nbig > 0) {
    const int CL = plan->adam_cluster;
    const int ncl = std::min(plan->adam_clusters, nbig);
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(ncl * CL);
    cfg.blockDim = dim3(kAdamThreads);
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = CL;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    cudaError_t e = cudaLaunchKernelEx(&cfg, adam_big_kernel<GT>, qb,
                                       ws_ptr<int32_t>(plan, plan->layout.big), nbig, ncl, g,
                                       d_factor, master, mq, vq, m_scale, v_scale, bf, k);
    if (e != cudaSuccess) return cuda_fail(e, "vsf_adam8_step (blocks)");
  }
  const int nsmall = (int)plan->small_blocks.size();
  if (nsmall > 0) {
    const int per = kSmallThreads / 32;
    adam_small_kernel<GT><<<(nsmall + per - 1) / per, kSmallThreads, 0, st>>>(
        qb, ws_ptr<int32_t>(plan, plan->layout.small), nsmall, g, d_factor, master, mq, vq,
        m_scale, v_scale, bf, k);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return cuda_fail(e, "vsf_adam8_step (element chunks)");
  }
  return VSF_OK;
}

}  // namespace
}  // namespace vsf

using namespace vsf;

extern "C" {

vsf_status vsf_plan_upload(vsf_plan* plan, void* d_workspace, size_t bytes, void* stream) {
  if (plan == nullptr || d_workspace == nullptr) return fail(VSF_ERR_ARG, "vsf_plan_upload: NULL");
  if (misaligned(d_workspace)) return fail(VSF_ERR_ALIGN, "vsf_plan_upload: workspace alignment");
  if (bytes < plan->layout.bytes) return fail(VSF_ERR_ARG, "vsf_plan_upload: workspace too small");
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  int dev = -1, sms = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (e != cudaSuccess) return cuda_fail(e, "vsf_plan_upload");

  // Copy grid: equal spans of the real elements, cut on 8-element multiples.
  const int grid = std::max(1, std::min(kMaxCopyGrid, sms * kCopyCtasPerSm));
  std::vector<CopySpan> spans(grid + 1);
  {
    std::vector<int64_t> starts(plan->n + 1, 0);
    for (int t = 0; t < plan->n; ++t) starts[t + 1] = starts[t] + plan->tensors[t].numel;
    int t = 0;
    for (int c = 0; c <= grid; ++c) {
      int64_t pos = (c == grid) ? plan->real : (plan->real / grid * c) / 8 * 8;
      while (t + 1 < plan->n && starts[t + 1] <= pos) ++t;
      if (c == grid) t = plan->n - 1;
      spans[c].tensor = t;
      spans[c].pad = 0;
      spans[c].elem = pos - starts[t];
    }
  }

  // Cluster size of the block kernel: smallest power of two keeping the
  // phase-1 bytes in flight (one block per cluster) within ~32 MB of L2.
  int occ = 0;
  e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, adam_big_kernel<uint16_t>,
                                                    kAdamThreads, 0);
  if (e != cudaSuccess) return cuda_fail(e, "vsf_plan_upload (occupancy)");
  occ = std::max(1, occ);
  int CL = 1;
  const double budget = 32.0 * 1024 * 1024;
  while (CL < kMaxCluster &&
         (double)sms * occ / CL * (double)plan->max_big_elems * 6.0 > budget)
    CL *= 2;
  int nclusters = sms * occ / CL;
  if (CL > 1) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(CL * 64);
    cfg.blockDim = dim3(kAdamThreads);
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = CL;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    int active = 0;
    e = cudaOccupancyMaxActiveClusters(&active, adam_big_kernel<uint16_t>, &cfg);
    if (e != cudaSuccess) return cuda_fail(e, "vsf_plan_upload (clusters)");
    if (active > 0) nclusters = active;
  }

  // Host image of the device tables; it lives in the plan so that the
  // asynchronous copy never reads freed memory.
  std::vector<unsigned char>& img = plan->upload_image;
  img.assign(plan->layout.spans + sizeof(CopySpan) * (grid + 1), 0);
  const DeviceLayout& L = plan->layout;
  for (int t = 0; t < plan->n; ++t) {
    std::memcpy(&img[L.tensor_off + 8 * t], &plan->tensors[t].offset, 8);
    std::memcpy(&img[L.tensor_numel + 8 * t], &plan->tensors[t].numel, 8);
  }
  if (!plan->qblocks.empty())
    std::memcpy(&img[L.qblocks], plan->qblocks.data(), sizeof(QBlock) * plan->qblocks.size());
  if (!plan->big_blocks.empty())
    std::memcpy(&img[L.big], plan->big_blocks.data(), 4 * plan->big_blocks.size());
  if (!plan->small_blocks.empty())
    std::memcpy(&img[L.small], plan->small_blocks.data(), 4 * plan->small_blocks.size());
  std::memcpy(&img[L.spans], spans.data(), sizeof(CopySpan) * spans.size());

  unsigned char* ws = static_cast<unsigned char*>(d_workspace);
  e = cudaMemsetAsync(ws, 0, plan->layout.bytes, st);
  if (e == cudaSuccess) e = cudaMemcpyAsync(ws, img.data(), img.size(), cudaMemcpyHostToDevice, st);
  if (e != cudaSuccess) return cuda_fail(e, "vsf_plan_upload (copy)");

  plan->d_ws = ws;
  plan->device = dev;
  plan->sm_count = sms;
  plan->copy_grid = grid;
  plan->adam_cluster = CL;
  plan->adam_clusters = std::max(1, nclusters);
  plan->uploaded = true;
  return VSF_OK;
}

vsf_status vsf_pack(const vsf_plan* plan, const void* const* grads, int32_t dtype,
                    void* packed_grad, void* stream) {
  vsf_status s = check_ready(plan, "vsf_pack");
  if (s != VSF_OK) return s;
  if (packed_grad == nullptr) return fail(VSF_ERR_ARG, "vsf_pack: NULL packed buffer");
  if (misaligned(packed_grad)) return fail(VSF_ERR_ALIGN, "vsf_pack: packed buffer alignment");
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (dtype == VSF_BF16) return launch_copy<uint16_t, kPack>(plan, grads, packed_grad, st, "vsf_pack");
  if (dtype == VSF_FP32) return launch_copy<float, kPack>(plan, grads, packed_grad, st, "vsf_pack");
  return fail(VSF_ERR_ARG, "vsf_pack: dtype must be VSF_BF16 or VSF_FP32");
}

vsf_status vsf_group_norm_scale(const vsf_plan* plan, const void* packed_grad, int32_t dtype,
                                const vsf_adam_hparams* hp, float* d_factor, double* d_norm,
                                void* stream) {
  vsf_status s = check_ready(plan, "vsf_group_norm_scale");
  if (s != VSF_OK) return s;
  if (hp == nullptr || d_factor == nullptr) return fail(VSF_ERR_ARG, "vsf_group_norm_scale: NULL");
  if (hp->world < 1) return fail(VSF_ERR_ARG, "vsf_group_norm_scale: world must be >= 1");
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (packed_grad != nullptr) {
    if (misaligned(packed_grad)) return fail(VSF_ERR_ALIGN, "vsf_group_norm_scale: alignment");
    if (dtype == VSF_BF16)
      s = launch_copy<uint16_t, kNormOnly>(plan, nullptr, const_cast<void*>(packed_grad), st,
                                           "vsf_group_norm_scale");
    else if (dtype == VSF_FP32)
      s = launch_copy<float, kNormOnly>(plan, nullptr, const_cast<void*>(packed_grad), st,
                                        "vsf_group_norm_scale");
    else
      return fail(VSF_ERR_ARG, "vsf_group_norm_scale: dtype must be VSF_BF16 or VSF_FP32");
    if (s != VSF_OK) return s;
  }
  norm_finalize_kernel<<<1, 256, 0, st>>>(
      reinterpret_cast<const double*>(plan->d_ws + plan->layout.partials), plan->copy_grid,
      hp->world, hp->max_norm, d_factor, d_norm);
  cudaError_t e = cudaGetLastError();
  return e == cudaSuccess ? VSF_OK : cuda_fail(e, "vsf_group_norm_scale");
}

vsf_status vsf_adam8_step(const vsf_plan* plan, const void* packed_grad, int32_t grad_dtype,
                          const float* d_factor, float* master, void* m_state, void* v_state,
                          float* m_scale, float* v_scale, uint16_t* packed_bf16,
                          const vsf_adam_hparams* hp, int32_t step, void* stream) {
  vsf_status s = check_ready(plan, "vsf_adam8_step");
  if (s != VSF_OK) return s;
  if (hp == nullptr || packed_grad == nullptr || d_factor == nullptr || master == nullptr ||
      m_state == nullptr || v_state == nullptr || packed_bf16 == nullptr)
    return fail(VSF_ERR_ARG, "vsf_adam8_step: NULL argument");
  if (hp->quantized && (m_scale == nullptr || v_scale == nullptr))
    return fail(VSF_ERR_ARG, "vsf_adam8_step: NULL scale array");
  if (step < 1) return fail(VSF_ERR_ARG, "vsf_adam8_step: step must be >= 1");
  if (misaligned(packed_grad) || misaligned(master) || misaligned(m_state) ||
      misaligned(v_state) || misaligned(packed_bf16) || misaligned(d_factor) ||
      (hp->quantized && (misaligned(m_scale) || misaligned(v_scale))))
    return fail(VSF_ERR_ALIGN, "vsf_adam8_step: pointer not 16-byte aligned");
  const AdamConsts k = make_consts(*hp, step);
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (grad_dtype == VSF_BF16)
    return launch_adam<uint16_t>(plan, packed_grad, d_factor, master, m_state, v_state, m_scale,
                                 v_scale, packed_bf16, k, hp->quantized != 0, st);
  if (grad_dtype == VSF_FP32)
    return launch_adam<float>(plan, packed_grad, d_factor, master, m_state, v_state, m_scale,
                              v_scale, packed_bf16, k, hp->quantized != 0, st);
  return fail(VSF_ERR_ARG, "vsf_adam8_step: grad_dtype must be VSF_BF16 or VSF_FP32");
}

vsf_status vsf_unpack(const vsf_plan* plan, const uint16_t* packed_bf16, void* const* params,
                      void* stream) {
  vsf_status s = check_ready(plan, "vsf_unpack");
  if (s != VSF_OK) return s;
  if (packed_bf16 == nullptr) return fail(VSF_ERR_ARG, "vsf_unpack: NULL packed buffer");
  if (misaligned(packed_bf16)) return fail(VSF_ERR_ALIGN, "vsf_unpack: packed buffer alignment");
  return launch_copy<uint16_t, kUnpack>(plan, const_cast<const void* const*>(params),
                                        const_cast<uint16_t*>(packed_bf16),
                                        static_cast<cudaStream_t>(stream), "vsf_unpack");
}

}  // extern "C"
