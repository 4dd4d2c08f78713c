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
// For a plan restricted to a rank window, the norm is split at its one
// cross-rank exchange: vsf_group_sumsq (this window's sum of squares) and
// vsf_group_scale_from_sumsq (the factor from the caller's total).
// Nothing here is a dense contraction: the kernels are HBM-bound streams
// (128-bit loads and stores, streaming cache hints, warp-shuffle reductions).
//
// Floating point: every fp32 operation of the AdamW update, the quantiser and
// the squared-norm accumulation is written with an explicit round-to-nearest
// intrinsic (__fmul_rn, __fadd_rn, __fdiv_rn, __fsqrt_rn, ...), which the
// compiler never contracts into an FMA, so each operation rounds once in the
// order written.
#include <cooperative_groups.h>
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cmath>
#include <cstring>
#include <algorithm>
#include <mutex>
#include <queue>
#include <string>
#include <utility>
#include <vector>

#include "bounds.cuh"
#include "vsf_internal.h"

namespace cg = cooperative_groups;

namespace vsf {
namespace {

constexpr int kCopyThreads = 256;
#ifndef VSF_COPY_CTAS_PER_SM
#define VSF_COPY_CTAS_PER_SM 16
#endif
constexpr int kCopyCtasPerSm = VSF_COPY_CTAS_PER_SM;
#ifndef VSF_COPY_UNROLL
#define VSF_COPY_UNROLL 8
#endif
constexpr int kCopyUnroll = VSF_COPY_UNROLL;  // 16-byte loads in flight per thread
constexpr int kMaxCluster = 8;
constexpr int kSmallThreads = 256;

struct TensorPtrs {
  const void* p[kMaxTensors];
};

// ------------------------------------------------------------------ helpers

__device__ __forceinline__ float bf16_to_f32(uint32_t h) { return __uint_as_float(h << 16); }

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

// x*x into the accumulator, with the FMA-recovered product error (fp32
// inputs).
__device__ __forceinline__ void acc_sq(DF& a, float x) {
  const float p = __fmul_rn(x, x);
  a.add(p);
  a.lo = __fadd_rn(a.lo, __fmaf_rn(x, x, -p));
}
// The same for a bf16 value: its square has at most 16 significant bits and
// is exact in fp32, so there is no product error to recover.
__device__ __forceinline__ void acc_sq_exact(DF& a, float x) { a.add(__fmul_rn(x, x)); }

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
    acc_sq_exact(acc, bf16_to_f32(w[i] & 0xffffu));
    acc_sq_exact(acc, bf16_to_f32(w[i] >> 16));
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
                                                            const int64_t* __restrict__ t_lo, const int64_t* __restrict__ t_hi,
                                                            const CopySpan* __restrict__ spans,
                                                            T* packed, double* partials, Bounds bd) {
  constexpr int V = 16 / sizeof(T);
  const CopySpan s0 = spans[blockIdx.x];
  const CopySpan s1 = spans[blockIdx.x + 1];
  DF acc;
  for (int t = s0.tensor; t <= s1.tensor; ++t) {
    const int64_t b = (t == s0.tensor) ? s0.elem : t_lo[t];
    const int64_t e = (t == s1.tensor) ? s1.elem : t_hi[t];
    if (b >= e || !in_bounds(bd, t_off[t] + b, t_off[t] + e)) continue;
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
      for (; k + (kCopyUnroll - 1) * kCopyThreads < nvec; k += kCopyUnroll * kCopyThreads) {
        uint4 r[kCopyUnroll];
#pragma unroll
        for (int u = 0; u < kCopyUnroll; ++u) r[u] = ld_stream(s + k + u * kCopyThreads);
#pragma unroll
        for (int u = 0; u < kCopyUnroll; ++u) {
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
  // An infinite running sum makes the error term NaN; keep the infinity.
  double v = warp_sum(isinf(acc.hi) ? (double)acc.hi : (double)acc.hi + (double)acc.lo);
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
// Fixed-order fp64 sum of n partials by one CTA of 256 threads; the result
// is valid in thread 0.
__device__ __forceinline__ double reduce_partials(const double* __restrict__ partials, int n) {
  __shared__ double red[256];
  double s = 0.0;
  for (int i = threadIdx.x; i < n; i += 256) s += partials[i];
  red[threadIdx.x] = s;
  __syncthreads();
  for (int w = 128; w > 0; w >>= 1) {
    if (threadIdx.x < w) red[threadIdx.x] += red[threadIdx.x + w];
    __syncthreads();
  }
  return red[0];
}

// norm = sqrt(sum of squares) / world; clip c = min(1, max_norm / (norm +
// 1e-6)) when max_norm is finite and positive; factor = fp32(c / world).
__device__ __forceinline__ void norm_factor(double sumsq, int world, double max_norm,
                                            float* d_factor, double* d_norm) {
  const double norm = sqrt(sumsq) / (double)world;
  double c = 1.0;
  if (isfinite(max_norm) && max_norm > 0.0) {
    const double r = max_norm / (norm + 1e-6);
    if (r < 1.0) c = r;
  }
  *d_factor = __double2float_rn(c / (double)world);
  if (d_norm) *d_norm = norm;
}

__global__ void __launch_bounds__(256) norm_finalize_kernel(const double* __restrict__ partials,
                                                            int n, int world, double max_norm,
                                                            float* d_factor, double* d_norm) {
  const double s = reduce_partials(partials, n);
  if (threadIdx.x == 0) norm_factor(s, world, max_norm, d_factor, d_norm);
}

__global__ void __launch_bounds__(256) sumsq_kernel(const double* __restrict__ partials, int n,
                                                    double* d_sumsq) {
  const double s = reduce_partials(partials, n);
  if (threadIdx.x == 0) *d_sumsq = s;
}

__global__ void factor_kernel(const double* __restrict__ d_sumsq, int world, double max_norm,
                              float* d_factor, double* d_norm) {
  norm_factor(*d_sumsq, world, max_norm, d_factor, d_norm);
}

#include "adam8.cuh"
#include "adam8_tma.cuh"

// The bulk-copy kernel instance of a plan's shape, with its block size and
// dynamic shared memory.
template <typename GT>
struct TmaLaunch {
  decltype(&adam_tma_kernel<GT, kTmaWideWarps>) fn;
  int threads;
  uint32_t smem;
};
template <typename GT>
TmaLaunch<GT> tma_launch(int warps) {
  if (warps == kTmaNarrowWarps)
    return {adam_tma_kernel<GT, kTmaNarrowWarps>, TmaShape<kTmaNarrowWarps>::threads,
            TmaLayout<GT, kTmaNarrowWarps>::total};
  return {adam_tma_kernel<GT, kTmaWideWarps>, TmaShape<kTmaWideWarps>::threads,
          TmaLayout<GT, kTmaWideWarps>::total};
}

// Fused group ops over every real element of a packed buffer (all tensors
// in one launch, over the copy spans): 0 zero, 1 scale by alpha, 2 add src.
// fp32 arithmetic with one rounding, then the buffer's type (bf16 RNE).
template <typename DT, typename ST, int kOp>
__device__ __forceinline__ DT group_elem(DT d, ST x, float alpha) {
  float r = 0.0f;
  if (kOp == 1) r = __fmul_rn(elem_f32(d), alpha);
  if (kOp == 2) r = __fadd_rn(elem_f32(d), elem_f32(x));
  if constexpr (sizeof(DT) == 2)
    return (DT)bf16_bits(r);
  else
    return r;
}

// E consecutive elements of a buffer, read and written as one vector access
// of E * sizeof(T) bytes (16 or 8), aligned to that size.
template <typename T, int E>
struct Group {
  static constexpr int kWords = E * (int)sizeof(T) / 4;
  alignas(16) T v[E];
  __device__ __forceinline__ void load(const T* p) {
    if constexpr (kWords == 4)
      *reinterpret_cast<uint4*>(v) = ld_stream(p);
    else
      *reinterpret_cast<uint2*>(v) = __ldcs(reinterpret_cast<const uint2*>(p));
  }
  __device__ __forceinline__ void store(T* p) const {
    if constexpr (kWords == 4)
      st_stream(p, *reinterpret_cast<const uint4*>(v));
    else
      __stcs(reinterpret_cast<uint2*>(p), *reinterpret_cast<const uint2*>(v));
  }
};

template <typename DT, typename ST, int kOp>
__global__ void __launch_bounds__(kCopyThreads) group_op_kernel(
    const int64_t* __restrict__ t_off, const int64_t* __restrict__ t_lo, const int64_t* __restrict__ t_hi,
    const CopySpan* __restrict__ spans, DT* dst, const ST* __restrict__ src, float alpha,
    Bounds bd) {
  // elements per vector group: 16 bytes of the wider type (8 bf16, 4 fp32)
  constexpr int E = 16 / (sizeof(DT) > sizeof(ST) ? sizeof(DT) : sizeof(ST));
  const CopySpan s0 = spans[blockIdx.x];
  const CopySpan s1 = spans[blockIdx.x + 1];
  for (int t = s0.tensor; t <= s1.tensor; ++t) {
    const int64_t b = (t == s0.tensor) ? s0.elem : t_lo[t];
    const int64_t e = (t == s1.tensor) ? s1.elem : t_hi[t];
    if (b >= e || !in_bounds(bd, t_off[t] + b, t_off[t] + e)) continue;
    const int64_t base = t_off[t];
    // buffer elements [x0, x1): scalar up to a multiple of E, then groups of
    // E (vector-aligned in both buffers), then the scalar tail
    const int64_t x0 = base + b, x1 = base + e;
    const int64_t v0 = min64(x1, (x0 + E - 1) / E * E), v1 = v0 + (x1 - v0) / E * E;
    for (int64_t x = x0 + threadIdx.x; x < v0; x += kCopyThreads)
      dst[x] = group_elem<DT, ST, kOp>(dst[x], kOp == 2 ? src[x] : ST(0), alpha);
    for (int64_t x = v0 + E * (int64_t)threadIdx.x; x < v1; x += E * kCopyThreads) {
      Group<DT, E> d;
      Group<ST, E> y;
      if (kOp != 0) d.load(dst + x);
      if (kOp == 2) y.load(src + x);
#pragma unroll
      for (int k = 0; k < E; ++k)
        d.v[k] = group_elem<DT, ST, kOp>(kOp != 0 ? d.v[k] : DT(0), kOp == 2 ? y.v[k] : ST(0), alpha);
      d.store(dst + x);
    }
    for (int64_t x = v1 + threadIdx.x; x < x1; x += kCopyThreads)
      dst[x] = group_elem<DT, ST, kOp>(dst[x], kOp == 2 ? src[x] : ST(0), alpha);
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

Bounds bounds_of(const vsf_plan* plan) {
  return Bounds{plan->total, reinterpret_cast<unsigned*>(plan->d_ws + plan->layout.error)};
}

// Step-t constants, each computed in double and rounded once to fp32
// (beta^t by t repeated multiplications); see adam8.cuh for the update.
AdamConsts make_consts(const vsf_adam_hparams& hp, int step) {
  double p1 = 1.0, p2 = 1.0;
  for (int i = 0; i < step; ++i) {
    p1 *= hp.beta1;
    p2 *= hp.beta2;
  }
  const double bc2s = std::sqrt(1.0 - p2);
  AdamConsts k;
  k.b1 = (float)hp.beta1;
  k.omb1 = (float)(1.0 - hp.beta1);
  k.b2 = (float)hp.beta2;
  k.omb2 = (float)(1.0 - hp.beta2);
  k.eps_hat = (float)(hp.eps * bc2s);
  k.decay = (float)(1.0 - hp.lr * hp.weight_decay);
  k.alpha = (float)(hp.lr * bc2s / (1.0 - p1));
  return k;
}

// Block-kernel variants: wide CTAs for clusters (one CTA per SM), narrower
// ones when a CTA owns whole blocks (two or more CTAs per SM).
#ifndef VSF_CLUSTER_THREADS
#define VSF_CLUSTER_THREADS 512
#define VSF_CLUSTER_MINB 1
#define VSF_CLUSTER_U1 4
#define VSF_CLUSTER_U2 2
#endif
#ifndef VSF_SOLO_THREADS
#define VSF_SOLO_THREADS 256
#define VSF_SOLO_MINB 4
#define VSF_SOLO_U1 2
#define VSF_SOLO_U2 1
#endif
constexpr int kClusterThreads = VSF_CLUSTER_THREADS;
constexpr int kSoloThreads = VSF_SOLO_THREADS;
template <typename GT>
constexpr auto kBlockKernelCluster = adam_block_kernel<GT, VSF_CLUSTER_THREADS, VSF_CLUSTER_MINB,
                                                       VSF_CLUSTER_U1, VSF_CLUSTER_U2>;
template <typename GT>
constexpr auto kBlockKernelSolo =
    adam_block_kernel<GT, VSF_SOLO_THREADS, VSF_SOLO_MINB, VSF_SOLO_U1, VSF_SOLO_U2>;

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
      ws_ptr<int64_t>(plan, plan->layout.tensor_lo),
      ws_ptr<int64_t>(plan, plan->layout.tensor_hi),
      ws_ptr<CopySpan>(plan, plan->layout.spans), static_cast<T*>(packed),
      reinterpret_cast<double*>(plan->d_ws + plan->layout.partials), bounds_of(plan));
  cudaError_t e = cudaGetLastError();
  return e == cudaSuccess ? VSF_OK : cuda_fail(e, who);
}

// cuTensorMapEncodeTiled through the runtime's driver entry point (no link
// against libcuda).
PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess)
      p = nullptr;
    return reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  }();
  return fn;
}

// The tile tensors' tensor maps for these arrays, re-encoded only when the
// pointers or the gradient type change since the previous call.
vsf_status tile_maps(const vsf_plan* plan, const void* grad, int grad_dtype, const void* mq,
                     const void* vq, const void* master, TileMaps* out) {
  std::memset(out, 0, sizeof(*out));
  out->count = (int32_t)plan->tile_maps.size();
  if (out->count == 0) return VSF_OK;
  std::lock_guard<std::mutex> lock(plan->maps_mu);
  const void* key[5] = {grad, mq, vq, master, nullptr};
  if (plan->maps_dtype == grad_dtype && std::memcmp(plan->maps_key, key, sizeof(key)) == 0 &&
      plan->maps_blob.size() == sizeof(TileMaps)) {
    std::memcpy(out, plan->maps_blob.data(), sizeof(TileMaps));
    return VSF_OK;
  }
  PFN_cuTensorMapEncodeTiled_v12000 encode = tensor_map_encoder();
  if (encode == nullptr) return fail(VSF_ERR_CUDA, "cuTensorMapEncodeTiled is unavailable");
  const CUtensorMapDataType gtype =
      grad_dtype == VSF_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT32;
  const int gsize = grad_dtype == VSF_BF16 ? 2 : 4;
  const void* arrays[4] = {grad, mq, vq, master};
  const CUtensorMapDataType types[4] = {gtype, CU_TENSOR_MAP_DATA_TYPE_UINT8,
                                        CU_TENSOR_MAP_DATA_TYPE_UINT8,
                                        CU_TENSOR_MAP_DATA_TYPE_FLOAT32};
  const int sizes[4] = {gsize, 1, 1, 4};
  for (int i = 0; i < out->count; ++i) {
    const TileMapInfo& mi = plan->tile_maps[i];
    out->tensor[i] = mi.tensor;
    for (int a = 0; a < 4; ++a) {
      cuuint64_t dims[2] = {(cuuint64_t)mi.cols, (cuuint64_t)mi.rows};
      cuuint64_t strides[1] = {(cuuint64_t)mi.cols * sizes[a]};
      cuuint32_t box[2] = {(cuuint32_t)mi.box_cols, (cuuint32_t)mi.box_rows};
      cuuint32_t estr[2] = {1, 1};
      void* addr = const_cast<char*>(static_cast<const char*>(arrays[a])) + mi.offset * sizes[a];
      CUresult r = encode(&out->m[i][a], types[a], 2, addr, dims, strides, box, estr,
                          CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
                          CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
      if (r != CUDA_SUCCESS)
        return fail(VSF_ERR_CUDA, "cuTensorMapEncodeTiled failed (" + std::to_string((int)r) + ")");
    }
  }
  plan->maps_blob.assign(reinterpret_cast<const unsigned char*>(out),
                         reinterpret_cast<const unsigned char*>(out) + sizeof(TileMaps));
  std::memcpy(plan->maps_key, key, sizeof(key));
  plan->maps_dtype = grad_dtype;
  return VSF_OK;
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
        ws_ptr<int64_t>(plan, plan->layout.tensor_lo),
      ws_ptr<int64_t>(plan, plan->layout.tensor_hi),
        ws_ptr<CopySpan>(plan, plan->layout.spans), g, d_factor, master,
        static_cast<float*>(m_state), static_cast<float*>(v_state), bf, k);
    cudaError_t e = cudaGetLastError();
    return e == cudaSuccess ? VSF_OK : cuda_fail(e, "vsf_adam8_step");
  }
  int8_t* mq = static_cast<int8_t*>(m_state);
  uint8_t* vq = static_cast<uint8_t*>(v_state);
  // Tensor maps before any launch: an encoding error must not leave the
  // step half applied.
  const int ntma = (int)plan->tma_blocks.size();
  TileMaps maps;
  if (ntma > 0) {
    vsf_status ms = tile_maps(plan, grad, sizeof(GT) == 2 ? VSF_BF16 : VSF_FP32, m_state, v_state,
                              master, &maps);
    if (ms != VSF_OK) return ms;
  }
  // Element chunks first: a short kernel that lets the bulk-copy kernel start
  // while it runs (the two touch disjoint blocks).
  const int nsmall = (int)plan->small_blocks.size();
  if (nsmall > 0) {
    const int per = kSmallThreads / 32;
    adam_small_kernel<GT><<<(nsmall + per - 1) / per, kSmallThreads, 0, st>>>(
        qb, ws_ptr<int32_t>(plan, plan->layout.small), nsmall, g, d_factor, master, mq, vq,
        m_scale, v_scale, bf, k);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return cuda_fail(e, "vsf_adam8_step (element chunks)");
  }
  if (ntma > 0) {
    const int CL = plan->tma_cluster;
    const int ncl = std::min(plan->tma_clusters, ntma);
    const TmaLaunch<GT> tl = tma_launch<GT>(plan->tma_warps);
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(ncl * CL);
    cfg.blockDim = dim3(tl.threads);
    cfg.dynamicSmemBytes = tl.smem;
    cfg.stream = st;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = CL;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    // programmatic serialization only right behind the element-chunk kernel
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[1].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = nsmall > 0 ? 2 : 1;
    cudaError_t e = cudaLaunchKernelEx(
        &cfg, tl.fn, maps, qb, ws_ptr<int32_t>(plan, plan->layout.tma),
        ws_ptr<int32_t>(plan, plan->layout.tma_k), ws_ptr<int32_t>(plan, plan->layout.tma_start),
        g,
        d_factor, master, mq, vq, m_scale, v_scale, bf, k,
        reinterpret_cast<unsigned*>(plan->d_ws + plan->layout.error));
    if (e != cudaSuccess) return cuda_fail(e, "vsf_adam8_step (bulk-copy blocks)");
  }
  const int nbig = (int)plan->big_blocks.size();
  if (nbig > 0) {
    const int CL = plan->adam_cluster;
    const int ncl = std::min(plan->adam_clusters, nbig);
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(ncl * CL);
    cfg.blockDim = dim3(CL > 1 ? kClusterThreads : kSoloThreads);
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = CL;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    cudaError_t e = cudaLaunchKernelEx(&cfg, CL > 1 ? kBlockKernelCluster<GT> : kBlockKernelSolo<GT>,
                                       qb, ws_ptr<int32_t>(plan, plan->layout.big), nbig, ncl, g,
                                       d_factor, master, mq, vq, m_scale, v_scale, bf, k);
    if (e != cudaSuccess) return cuda_fail(e, "vsf_adam8_step (blocks)");
  }
  return VSF_OK;
}

}  // namespace
}  // namespace vsf

using namespace vsf;

extern "C" {

vsf_status vsf_plan_upload(vsf_plan* plan, void* d_workspace, size_t bytes, void* stream) {
  vsf::Range nvtx_range("vsf_plan_upload");
  if (plan == nullptr || d_workspace == nullptr) return fail(VSF_ERR_ARG, "vsf_plan_upload: NULL");
  if (misaligned(d_workspace)) return fail(VSF_ERR_ALIGN, "vsf_plan_upload: workspace alignment");
  if (bytes < plan->layout.bytes) return fail(VSF_ERR_ARG, "vsf_plan_upload: workspace too small");
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  int dev = -1, sms = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (e != cudaSuccess) return cuda_fail(e, "vsf_plan_upload");

  // Copy grid: equal spans of the real elements inside the rank window
  // (each tensor's [lo, hi)), cut on 8-element multiples. kCopyCtasPerSm
  // CTAs per SM for large buffers; a small buffer gets at least one full
  // unrolled pass of 16-byte loads per CTA instead of thousands of nearly
  // empty CTAs (and as many partials for the norm to reduce).
  constexpr int64_t kMinCopyElems = (int64_t)kCopyUnroll * kCopyThreads * 8;
  const int64_t by_work = (plan->real + kMinCopyElems - 1) / kMinCopyElems;
  const int grid = (int)std::max<int64_t>(
      1, std::min<int64_t>(by_work, std::min(kMaxCopyGrid, sms * kCopyCtasPerSm)));
  std::vector<CopySpan> spans(grid + 1);
  {
    std::vector<int64_t> starts(plan->n + 1, 0);
    for (int t = 0; t < plan->n; ++t)
      starts[t + 1] = starts[t] + (plan->tensors[t].hi - plan->tensors[t].lo);
    int t = 0;
    for (int c = 0; c <= grid; ++c) {
      int64_t pos = (c == grid) ? plan->real : (plan->real / grid * c) / 8 * 8;
      while (t + 1 < plan->n && starts[t + 1] <= pos) ++t;
      if (c == grid) t = plan->n - 1;
      spans[c].tensor = t;
      spans[c].pad = 0;
      spans[c].elem = plan->tensors[t].lo + (pos - starts[t]);
    }
  }

  // Cluster size of the block kernel: the smallest of 1, 2, 4, 8 (3 and 6
  // split a block's chunks unevenly and measured slower) that keeps
  // the phase-1 bytes in flight (one block per active cluster, 4 B per
  // element) within the L2 budget (128 MB of the 126 MB L2 measured best:
  // phase 2 re-reads the newest part of each block first, and smaller
  // clusters let every SM work), so that phase 2's re-read hits.
#ifndef VSF_L2_BUDGET_MB
#define VSF_L2_BUDGET_MB 128
#endif
  const double budget = VSF_L2_BUDGET_MB * 1024.0 * 1024.0;
  int CL = 0, nclusters = 0;
  for (int cand = 1; cand <= kMaxCluster; cand *= 2) {
    int active = 0;
    if (cand == 1) {
      int occ = 0;
      e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, kBlockKernelSolo<uint16_t>,
                                                        kSoloThreads, 0);
      if (e != cudaSuccess) return cuda_fail(e, "vsf_plan_upload (occupancy)");
      active = std::max(1, occ) * sms;
    } else {
      cudaLaunchConfig_t cfg = {};
      cfg.gridDim = dim3(cand * 64);
      cfg.blockDim = dim3(kClusterThreads);
      cudaLaunchAttribute attr[1];
      attr[0].id = cudaLaunchAttributeClusterDimension;
      attr[0].val.clusterDim.x = cand;
      attr[0].val.clusterDim.y = 1;
      attr[0].val.clusterDim.z = 1;
      cfg.attrs = attr;
      cfg.numAttrs = 1;
      e = cudaOccupancyMaxActiveClusters(&active, kBlockKernelCluster<uint16_t>, &cfg);
      if (e != cudaSuccess) return cuda_fail(e, "vsf_plan_upload (clusters)");
      active = std::max(1, active);
    }
    CL = cand;
    nclusters = active;
    if ((double)active * (double)plan->max_big_elems * 4.0 <= budget) break;
  }

  // Bulk-copy kernel: 16 / warps CTAs per SM (their rings take ~200 KB of
  // shared memory together). Its cluster size: the smallest power of two for
  // which the phase-1 bytes of the units in flight (one unit per cluster,
  // 4 B per element) stay within half the L2, with units counted at their
  // element-weighted mean size (the size of the unit an average element
  // belongs to), as the clusters work through units of every size. Measured
  // on the four large workloads: 53-56 MB in flight kept every phase-2
  // re-read in L2 or close to it; 80 MB (DSv3 block in clusters of 1) and
  // 110 MB (Llama layer in clusters of 1, MoE layer in clusters of 2) ran
  // 1.5-10% slower than the next cluster size up, and a cluster size beyond
  // the first that fits lost again (shorter shares, wider exchange).
#ifndef VSF_BULK_L2_BUDGET_MB
#define VSF_BULK_L2_BUDGET_MB 64
#endif
  const double tma_budget = VSF_BULK_L2_BUDGET_MB * 1024.0 * 1024.0;
  int tma_CL = 1, tma_ncl = 1;
  {
    for (int w : {kTmaWideWarps, kTmaNarrowWarps}) {
      const TmaLaunch<uint16_t> a = tma_launch<uint16_t>(w);
      const TmaLaunch<float> b = tma_launch<float>(w);
      e = cudaFuncSetAttribute(a.fn, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)a.smem);
      if (e == cudaSuccess)
        e = cudaFuncSetAttribute(b.fn, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)b.smem);
      if (e != cudaSuccess) return cuda_fail(e, "vsf_plan_upload (shared memory size)");
    }
    const TmaLaunch<uint16_t> tl = tma_launch<uint16_t>(plan->tma_warps);
    for (int cand = 1; cand <= kMaxCluster; cand *= 2) {
      cudaLaunchConfig_t cfg = {};
      cfg.gridDim = dim3(cand * 64);
      cfg.blockDim = dim3(tl.threads);
      cfg.dynamicSmemBytes = tl.smem;
      cudaLaunchAttribute attr[1];
      attr[0].id = cudaLaunchAttributeClusterDimension;
      attr[0].val.clusterDim.x = cand;
      attr[0].val.clusterDim.y = 1;
      attr[0].val.clusterDim.z = 1;
      cfg.attrs = attr;
      cfg.numAttrs = 1;
      int active = 0;
      e = cudaOccupancyMaxActiveClusters(&active, tl.fn, &cfg);
      if (e != cudaSuccess) return cuda_fail(e, "vsf_plan_upload (bulk-copy clusters)");
      tma_CL = cand;
      tma_ncl = std::max(1, active);
      if ((double)tma_ncl * plan->tma_unit_mean * 4.0 <= tma_budget) break;
    }
  }

  // Host image of the device tables; it lives in the plan so that the
  // asynchronous copy never reads freed memory.
  std::vector<unsigned char>& img = plan->upload_image;
  img.assign(plan->layout.spans + sizeof(CopySpan) * (grid + 1), 0);
  const DeviceLayout& L = plan->layout;
  for (int t = 0; t < plan->n; ++t) {
    const int64_t off = plan->tensors[t].offset - (int64_t)plan->rank_begin * plan->S;
    std::memcpy(&img[L.tensor_off + 8 * t], &off, 8);
    std::memcpy(&img[L.tensor_lo + 8 * t], &plan->tensors[t].lo, 8);
    std::memcpy(&img[L.tensor_hi + 8 * t], &plan->tensors[t].hi, 8);
  }
  if (!plan->qblocks.empty())
    std::memcpy(&img[L.qblocks], plan->qblocks.data(), sizeof(QBlock) * plan->qblocks.size());
  if (!plan->big_blocks.empty())
    std::memcpy(&img[L.big], plan->big_blocks.data(), 4 * plan->big_blocks.size());
  if (!plan->small_blocks.empty())
    std::memcpy(&img[L.small], plan->small_blocks.data(), 4 * plan->small_blocks.size());
  if (!plan->tma_blocks.empty()) {
    // Bulk-copy units per cluster by longest-processing-time greedy over
    // their element counts: units by size, largest first, each to the
    // cluster with the least work so far. Cluster c then runs its units
    // from list[starts[c]] to list[starts[c+1]-1] in tensor order, so that
    // the clusters run a mix of unit sizes at any time. With the units dealt
    // round-robin, the clusters that drew more large units ran up to ~10%
    // longer than the mean (Llama layer); running every cluster's largest
    // units first put all the large units in flight at once, and their
    // phase-1 data no longer fit in L2 (1.3B model: 5% slower).
    const int ntma = (int)plan->tma_blocks.size();
    const int ncl = std::min(tma_ncl, ntma);
    if (ncl > kMaxCopyGrid) return fail(VSF_ERR_STATE, "vsf_plan_upload: too many clusters");
    std::vector<int64_t> size(ntma);
    for (int u = 0; u < ntma; ++u) {
      const QBlock& b = plan->qblocks[plan->tma_blocks[u]];
      size[u] = (int64_t)b.nrows * b.ncols * plan->tma_tiles[u];
    }
    std::vector<int> by_size(ntma);
    for (int u = 0; u < ntma; ++u) by_size[u] = u;
    std::stable_sort(by_size.begin(), by_size.end(),
                     [&](int a, int b) { return size[a] > size[b]; });
    using Load = std::pair<int64_t, int>;  // (elements so far, cluster)
    std::priority_queue<Load, std::vector<Load>, std::greater<Load>> heap;
    for (int c = 0; c < ncl; ++c) heap.push({0, c});
    std::vector<std::vector<int>> mine(ncl);
    for (int u : by_size) {
      Load l = heap.top();
      heap.pop();
      mine[l.second].push_back(u);
      heap.push({l.first + size[u], l.second});
    }
    std::vector<int32_t> list, ks, starts(ncl + 1, 0);
    list.reserve(ntma);
    ks.reserve(ntma);
    for (int c = 0; c < ncl; ++c) {
      std::vector<int>& mc = mine[c];
      std::sort(mc.begin(), mc.end());  // tensor order ...
      if (!mc.empty())                  // ... from a point of its own
        std::rotate(mc.begin(), mc.begin() + (size_t)c * mc.size() / ncl, mc.end());
      for (int u : mc) {
        list.push_back(plan->tma_blocks[u]);
        ks.push_back(plan->tma_tiles[u]);
      }
      starts[c + 1] = (int32_t)list.size();
    }
    std::memcpy(&img[L.tma], list.data(), 4 * list.size());
    std::memcpy(&img[L.tma_k], ks.data(), 4 * ks.size());
    std::memcpy(&img[L.tma_start], starts.data(), 4 * starts.size());
  }
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
  plan->tma_cluster = tma_CL;
  plan->tma_clusters = tma_ncl;
  const vsf_status lanes = muon_lanes_create(plan);
  if (lanes != VSF_OK) return lanes;
  plan->uploaded = true;
  return VSF_OK;
}

vsf_status vsf_pack(const vsf_plan* plan, const void* const* grads, int32_t dtype,
                    void* packed_grad, void* stream) {
  vsf::Range nvtx_range("vsf_pack");
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
  vsf::Range nvtx_range("vsf_group_norm_scale");
  vsf_status s = check_ready(plan, "vsf_group_norm_scale");
  if (s != VSF_OK) return s;
  if (plan->rank_begin != 0 || plan->rank_end != plan->m)
    return fail(VSF_ERR_STATE,
                "vsf_group_norm_scale: the plan covers a rank window; use vsf_group_sumsq, "
                "sum across windows, then vsf_group_scale_from_sumsq");
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

vsf_status vsf_group_sumsq(const vsf_plan* plan, const void* packed_grad, int32_t dtype,
                           double* d_sumsq, void* stream) {
  vsf::Range nvtx_range("vsf_group_sumsq");
  vsf_status s = check_ready(plan, "vsf_group_sumsq");
  if (s != VSF_OK) return s;
  if (d_sumsq == nullptr) return fail(VSF_ERR_ARG, "vsf_group_sumsq: NULL d_sumsq");
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (packed_grad != nullptr) {
    if (misaligned(packed_grad)) return fail(VSF_ERR_ALIGN, "vsf_group_sumsq: alignment");
    if (dtype == VSF_BF16)
      s = launch_copy<uint16_t, kNormOnly>(plan, nullptr, const_cast<void*>(packed_grad), st,
                                           "vsf_group_sumsq");
    else if (dtype == VSF_FP32)
      s = launch_copy<float, kNormOnly>(plan, nullptr, const_cast<void*>(packed_grad), st,
                                        "vsf_group_sumsq");
    else
      return fail(VSF_ERR_ARG, "vsf_group_sumsq: dtype must be VSF_BF16 or VSF_FP32");
    if (s != VSF_OK) return s;
  }
  sumsq_kernel<<<1, 256, 0, st>>>(reinterpret_cast<const double*>(plan->d_ws + plan->layout.partials),
                                  plan->copy_grid, d_sumsq);
  cudaError_t e = cudaGetLastError();
  return e == cudaSuccess ? VSF_OK : cuda_fail(e, "vsf_group_sumsq");
}

vsf_status vsf_selftest_wait_timeout(unsigned* d_err, uint64_t limit_ns, void* stream) {
  if (d_err == nullptr) return fail(VSF_ERR_ARG, "vsf_selftest_wait_timeout: NULL error word");
  if (limit_ns > 1000000000ull)
    return fail(VSF_ERR_ARG, "vsf_selftest_wait_timeout: limit above 1 s");
  wait_selftest_kernel<<<1, 32, 0, static_cast<cudaStream_t>(stream)>>>(d_err, limit_ns);
  cudaError_t e = cudaGetLastError();
  return e == cudaSuccess ? VSF_OK : cuda_fail(e, "vsf_selftest_wait_timeout");
}

vsf_status vsf_group_scale_from_sumsq(const double* d_sumsq, const vsf_adam_hparams* hp,
                                      float* d_factor, double* d_norm, void* stream) {
  vsf::Range nvtx_range("vsf_group_scale_from_sumsq");
  if (d_sumsq == nullptr || hp == nullptr || d_factor == nullptr)
    return fail(VSF_ERR_ARG, "vsf_group_scale_from_sumsq: NULL argument");
  if (hp->world < 1) return fail(VSF_ERR_ARG, "vsf_group_scale_from_sumsq: world must be >= 1");
  factor_kernel<<<1, 1, 0, static_cast<cudaStream_t>(stream)>>>(d_sumsq, hp->world, hp->max_norm,
                                                                 d_factor, d_norm);
  cudaError_t e = cudaGetLastError();
  return e == cudaSuccess ? VSF_OK : cuda_fail(e, "vsf_group_scale_from_sumsq");
}

vsf_status vsf_adam8_step(const vsf_plan* plan, const void* packed_grad, int32_t grad_dtype,
                          const float* d_factor, float* master, void* m_state, void* v_state,
                          float* m_scale, float* v_scale, uint16_t* packed_bf16,
                          const vsf_adam_hparams* hp, int32_t step, void* stream) {
  vsf::Range nvtx_range("vsf_adam8_step");
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
  AdamConsts k = make_consts(*hp, step);
  k.bd = bounds_of(plan);
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
  vsf::Range nvtx_range("vsf_unpack");
  vsf_status s = check_ready(plan, "vsf_unpack");
  if (s != VSF_OK) return s;
  if (packed_bf16 == nullptr) return fail(VSF_ERR_ARG, "vsf_unpack: NULL packed buffer");
  if (misaligned(packed_bf16)) return fail(VSF_ERR_ALIGN, "vsf_unpack: packed buffer alignment");
  return launch_copy<uint16_t, kUnpack>(plan, const_cast<const void* const*>(params),
                                        const_cast<uint16_t*>(packed_bf16),
                                        static_cast<cudaStream_t>(stream), "vsf_unpack");
}

}  // extern "C"

// ------------------------------------------------------------------ copy ceiling

namespace vsf {
namespace {

constexpr int kCeilThreads = 512;
constexpr int kCeilUnroll = 8;

// dst[i] = src[i] over n 16-byte words: each thread keeps kCeilUnroll
// streaming loads in flight, grid-stride over the whole range.
__global__ void __launch_bounds__(kCeilThreads) device_copy_kernel(uint4* __restrict__ dst,
                                                                   const uint4* __restrict__ src,
                                                                   int64_t n) {
  const int64_t stride = (int64_t)gridDim.x * kCeilThreads;
  int64_t i = (int64_t)blockIdx.x * kCeilThreads + threadIdx.x;
  for (; i + (kCeilUnroll - 1) * stride < n; i += kCeilUnroll * stride) {
    uint4 r[kCeilUnroll];
#pragma unroll
    for (int u = 0; u < kCeilUnroll; ++u) r[u] = ld_stream(src + i + u * stride);
#pragma unroll
    for (int u = 0; u < kCeilUnroll; ++u) st_stream(dst + i + u * stride, r[u]);
  }
  for (; i < n; i += stride) st_stream(dst + i, ld_stream(src + i));
}

}  // namespace
}  // namespace vsf

extern "C" vsf_status vsf_device_copy(void* dst, const void* src, size_t bytes, void* stream) {
  using namespace vsf;
  if (dst == nullptr || src == nullptr) return fail(VSF_ERR_ARG, "vsf_device_copy: NULL pointer");
  if (bytes % 16 != 0) return fail(VSF_ERR_ARG, "vsf_device_copy: bytes not a multiple of 16");
  if (misaligned(dst) || misaligned(src))
    return fail(VSF_ERR_ALIGN, "vsf_device_copy: pointer not 16-byte aligned");
  if (bytes == 0) return VSF_OK;
  int dev = -1, sms = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (e != cudaSuccess) return cuda_fail(e, "vsf_device_copy");
  device_copy_kernel<<<sms * 4, kCeilThreads, 0, static_cast<cudaStream_t>(stream)>>>(
      static_cast<uint4*>(dst), static_cast<const uint4*>(src), (int64_t)(bytes / 16));
  e = cudaGetLastError();
  return e == cudaSuccess ? VSF_OK : cuda_fail(e, "vsf_device_copy");
}

// ------------------------------------------------------------------ fused group ops

namespace vsf {
namespace {

template <typename DT, typename ST, int kOp>
vsf_status launch_group(const vsf_plan* plan, void* dst, const void* src, float alpha,
                        cudaStream_t st, const char* who) {
  group_op_kernel<DT, ST, kOp><<<plan->copy_grid, kCopyThreads, 0, st>>>(
      ws_ptr<int64_t>(plan, plan->layout.tensor_off),
      ws_ptr<int64_t>(plan, plan->layout.tensor_lo),
      ws_ptr<int64_t>(plan, plan->layout.tensor_hi),
      ws_ptr<CopySpan>(plan, plan->layout.spans), static_cast<DT*>(dst),
      static_cast<const ST*>(src), alpha, bounds_of(plan));
  cudaError_t e = cudaGetLastError();
  return e == cudaSuccess ? VSF_OK : cuda_fail(e, who);
}

}  // namespace
}  // namespace vsf

extern "C" {

vsf_status vsf_group_zero(const vsf_plan* plan, void* buf, int32_t dtype, void* stream) {
  vsf::Range nvtx_range("vsf_group_zero");
  using namespace vsf;
  vsf_status s = check_ready(plan, "vsf_group_zero");
  if (s != VSF_OK) return s;
  if (buf == nullptr) return fail(VSF_ERR_ARG, "vsf_group_zero: NULL buffer");
  if (misaligned(buf)) return fail(VSF_ERR_ALIGN, "vsf_group_zero: alignment");
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (dtype == VSF_BF16) return launch_group<uint16_t, uint16_t, 0>(plan, buf, nullptr, 0.f, st, "vsf_group_zero");
  if (dtype == VSF_FP32) return launch_group<float, float, 0>(plan, buf, nullptr, 0.f, st, "vsf_group_zero");
  return fail(VSF_ERR_ARG, "vsf_group_zero: dtype must be VSF_BF16 or VSF_FP32");
}

vsf_status vsf_group_scale(const vsf_plan* plan, void* buf, int32_t dtype, float alpha,
                           void* stream) {
  vsf::Range nvtx_range("vsf_group_scale");
  using namespace vsf;
  vsf_status s = check_ready(plan, "vsf_group_scale");
  if (s != VSF_OK) return s;
  if (buf == nullptr) return fail(VSF_ERR_ARG, "vsf_group_scale: NULL buffer");
  if (misaligned(buf)) return fail(VSF_ERR_ALIGN, "vsf_group_scale: alignment");
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (dtype == VSF_BF16) return launch_group<uint16_t, uint16_t, 1>(plan, buf, nullptr, alpha, st, "vsf_group_scale");
  if (dtype == VSF_FP32) return launch_group<float, float, 1>(plan, buf, nullptr, alpha, st, "vsf_group_scale");
  return fail(VSF_ERR_ARG, "vsf_group_scale: dtype must be VSF_BF16 or VSF_FP32");
}

vsf_status vsf_group_add(const vsf_plan* plan, void* dst, int32_t dst_dtype, const void* src,
                         int32_t src_dtype, void* stream) {
  vsf::Range nvtx_range("vsf_group_add");
  using namespace vsf;
  vsf_status s = check_ready(plan, "vsf_group_add");
  if (s != VSF_OK) return s;
  if (dst == nullptr || src == nullptr) return fail(VSF_ERR_ARG, "vsf_group_add: NULL buffer");
  if (misaligned(dst) || misaligned(src)) return fail(VSF_ERR_ALIGN, "vsf_group_add: alignment");
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const char* who = "vsf_group_add";
  if (dst_dtype == VSF_BF16 && src_dtype == VSF_BF16) return launch_group<uint16_t, uint16_t, 2>(plan, dst, src, 0.f, st, who);
  if (dst_dtype == VSF_FP32 && src_dtype == VSF_BF16) return launch_group<float, uint16_t, 2>(plan, dst, src, 0.f, st, who);
  if (dst_dtype == VSF_FP32 && src_dtype == VSF_FP32) return launch_group<float, float, 2>(plan, dst, src, 0.f, st, who);
  if (dst_dtype == VSF_BF16 && src_dtype == VSF_FP32) return launch_group<uint16_t, float, 2>(plan, dst, src, 0.f, st, who);
  return fail(VSF_ERR_ARG, "vsf_group_add: dtypes must be VSF_BF16 or VSF_FP32");
}

}  // extern "C"

// ------------------------------------------------------------------ group norm without allocation
//
// For callers that cannot allocate device memory at the point where they need
// the gradient norm: a hook that runs inside a framework's caching allocator
// (its out-of-memory or reclaim path, where asking for memory would recurse
// into the allocator), a runtime that owns the whole device memory budget and
// forbids raw cudaMalloc, or latency-critical code that cannot afford the
// device synchronisation cudaMalloc and cudaFree may imply. Everything the
// computation needs beyond its inputs and outputs lives in the file-scope
// array below, which every device that loads the library holds until the
// process exits.

namespace vsf {
namespace {

constexpr int kStaticPartials = 1024;     // at most this many CTAs, one partial each
constexpr int kStaticMaxTensors = 1024;   // tensors per call (kernel parameter space)

// Per-CTA partial sums of squares of the allocation-free norm. 8 KB.
static __device__ __align__(256) double g_static_partials[kStaticPartials];

struct StaticNormArgs {
  const void* p[kStaticMaxTensors];
  int64_t prefix[kStaticMaxTensors + 1];  // prefix[t] = elements before tensor t
  int32_t n;
};

// CTA c sums g^2 over elements [c*N/G, (c+1)*N/G) of the concatenated tensors
// (cut on 8-element multiples), like the copy kernel's norm pass, and writes
// its partial to partials[c]. Every slot in [0, gridDim.x) is written.
template <typename T>
__global__ void __launch_bounds__(kCopyThreads) sumsq_static_kernel(StaticNormArgs a,
                                                                    double* partials) {
  constexpr int V = 16 / sizeof(T);
  const int64_t N = a.prefix[a.n];
  const int64_t G = gridDim.x;
  const int64_t lo = (N / G * blockIdx.x) / 8 * 8;
  const int64_t hi = blockIdx.x + 1 == G ? N : (N / G * (blockIdx.x + 1)) / 8 * 8;
  DF acc;
  // first tensor with prefix[t + 1] > lo
  int t0 = 0, t1 = a.n;
  while (t0 < t1) {
    const int mid = (t0 + t1) / 2;
    if (a.prefix[mid + 1] <= lo) t0 = mid + 1; else t1 = mid;
  }
  for (int t = t0; t < a.n && a.prefix[t] < hi; ++t) {
    const int64_t b = max(lo, a.prefix[t]) - a.prefix[t];
    const int64_t e = min(hi, a.prefix[t + 1]) - a.prefix[t];
    const T* src = static_cast<const T*>(a.p[t]);
    int64_t i = b;
    if (((reinterpret_cast<uintptr_t>(src + b)) & 15) == 0) {
      const int64_t nvec = (e - b) / V;
      const uint4* s = reinterpret_cast<const uint4*>(src + b);
      for (int64_t k = threadIdx.x; k < nvec; k += kCopyThreads) sq_vec<T>(acc, ld_stream(s + k));
      i = b + nvec * V;
    }
    for (int64_t j = i + threadIdx.x; j < e; j += kCopyThreads) acc_sq(acc, elem_f32(src[j]));
  }
  __shared__ double red[kCopyThreads / 32];
  double v = warp_sum(isinf(acc.hi) ? (double)acc.hi : (double)acc.hi + (double)acc.lo);
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = v;
  __syncthreads();
  if (threadIdx.x == 0) {
    double s = 0.0;
    for (int w = 0; w < kCopyThreads / 32; ++w) s += red[w];
    partials[blockIdx.x] = s;
  }
}

std::mutex g_static_mu;
// Device address of g_static_partials per device, with the context it was
// looked up in: after a device reset the primary context (and with it the
// module and the array's address) is new, and the address is looked up again.
struct StaticAddr {
  CUcontext ctx = nullptr;
  double* ptr = nullptr;
};
StaticAddr g_static_addr[256];

using CtxGetCurrentFn = CUresult (*)(CUcontext*);
CtxGetCurrentFn ctx_get_current() {
  static CtxGetCurrentFn fn = [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 12000, cudaEnableDefault, &q) !=
            cudaSuccess ||
        q != cudaDriverEntryPointSuccess)
      p = nullptr;
    return reinterpret_cast<CtxGetCurrentFn>(p);
  }();
  return fn;
}

// Looks the array's device address up (with the device current) once per
// device and context; host code cannot use the symbol itself as a device
// pointer.
vsf_status static_partials(int dev, double** out) {
  if (dev < 0 || dev >= 256) return fail(VSF_ERR_ARG, "vsf_group_norm_scale_static: device id");
  CtxGetCurrentFn get_ctx = ctx_get_current();
  if (get_ctx == nullptr) return fail(VSF_ERR_CUDA, "cuCtxGetCurrent is unavailable");
  CUcontext ctx = nullptr;
  if (get_ctx(&ctx) != CUDA_SUCCESS || ctx == nullptr)
    return fail(VSF_ERR_CUDA, "vsf_group_norm_scale_static: no current context");
  std::lock_guard<std::mutex> lock(g_static_mu);
  StaticAddr& a = g_static_addr[dev];
  if (a.ptr == nullptr || a.ctx != ctx) {
    void* p = nullptr;
    cudaError_t e = cudaGetSymbolAddress(&p, g_static_partials);
    if (e != cudaSuccess) return cuda_fail(e, "vsf_group_norm_scale_static (symbol address)");
    a.ptr = static_cast<double*>(p);
    a.ctx = ctx;
  }
  *out = a.ptr;
  return VSF_OK;
}

}  // namespace
}  // namespace vsf

extern "C" vsf_status vsf_group_norm_scale_static(const void* const* grads, const int64_t* numel,
                                                  int32_t n, int32_t dtype,
                                                  const vsf_adam_hparams* hp, float* d_factor,
                                                  double* d_norm, void* stream) {
  using namespace vsf;
  Range nvtx_range("vsf_group_norm_scale_static");
  if (grads == nullptr || numel == nullptr || hp == nullptr || d_factor == nullptr)
    return fail(VSF_ERR_ARG, "vsf_group_norm_scale_static: NULL argument");
  if (n < 1 || n > kStaticMaxTensors)
    return fail(VSF_ERR_ARG, "vsf_group_norm_scale_static: n must be 1..1024 tensors, got " +
                                 std::to_string(n));
  if (hp->world < 1) return fail(VSF_ERR_ARG, "vsf_group_norm_scale_static: world must be >= 1");
  if (dtype != VSF_BF16 && dtype != VSF_FP32)
    return fail(VSF_ERR_ARG, "vsf_group_norm_scale_static: dtype must be VSF_BF16 or VSF_FP32");
  StaticNormArgs a;
  std::memset(&a, 0, sizeof(a));
  a.n = n;
  a.prefix[0] = 0;
  for (int t = 0; t < n; ++t) {
    if (grads[t] == nullptr || numel[t] < 1)
      return fail(VSF_ERR_ARG, "vsf_group_norm_scale_static: tensor " + std::to_string(t) +
                                   " is NULL or empty");
    if (misaligned(grads[t]))
      return fail(VSF_ERR_ALIGN, "vsf_group_norm_scale_static: tensor " + std::to_string(t) +
                                     " not 16-byte aligned");
    if (a.prefix[t] > INT64_MAX / 2 - numel[t])
      return fail(VSF_ERR_OVERFLOW, "vsf_group_norm_scale_static: too many elements");
    a.p[t] = grads[t];
    a.prefix[t + 1] = a.prefix[t] + numel[t];
  }
  int dev = -1, sms = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (e != cudaSuccess) return cuda_fail(e, "vsf_group_norm_scale_static");
  double* partials = nullptr;
  vsf_status s = static_partials(dev, &partials);
  if (s != VSF_OK) return s;
  const int grid = std::max(1, std::min(kStaticPartials, sms * 4));
  if (grid > kStaticPartials)  // the array bounds the grid, never the reverse
    return fail(VSF_ERR_ARG, "vsf_group_norm_scale_static: grid exceeds the static scratch");
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (dtype == VSF_BF16)
    sumsq_static_kernel<uint16_t><<<grid, kCopyThreads, 0, st>>>(a, partials);
  else
    sumsq_static_kernel<float><<<grid, kCopyThreads, 0, st>>>(a, partials);
  e = cudaGetLastError();
  if (e != cudaSuccess) return cuda_fail(e, "vsf_group_norm_scale_static (sum of squares)");
  norm_finalize_kernel<<<1, 256, 0, st>>>(partials, grid, hp->world, hp->max_norm, d_factor,
                                          d_norm);
  e = cudaGetLastError();
  return e == cudaSuccess ? VSF_OK : cuda_fail(e, "vsf_group_norm_scale_static (finalize)");
}
