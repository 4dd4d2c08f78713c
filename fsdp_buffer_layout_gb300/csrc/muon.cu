// muon.cu — distributed Muon on the planned buffer ("veScale-FSDP: Flexible and
// High-Performance FSDP at Scale (MLSys 2026)" summary page › 结构感知训练 case
// study › 分布式 Muon, Algorithm 2).
//
// On one GPU with all m virtual ranks in one buffer, the algorithm's steps map
// as follows:
//   SelectRoot()          host: longest-processing-time greedy over the
//                         Newton-Schulz FLOPs of every matrix tensor
//                         (vsf_muon_select_roots);
//   Redistribute(u, root) zero-copy: a tensor is contiguous in the buffer, so
//                         the root's "whole matrix" is a view of it;
//   Newton-Schulz         on the root: 5 quintic iterations, 3 tensor-core
//                         products each (this library's tcgen05 kernel,
//                         ns_gemm.cuh: bf16 operands, fp32 accumulation in
//                         TMEM, the two symmetric products on half their
//                         tiles), batched over a tensor's matrices;
//   Redistribute back     zero-copy again; the element-wise update writes the
//                         ragged shards in place.
// Matrices of one shape from every tensor are batched into the same launches
// (in chunks), so that many small matrices still fill the GPU.
// Own kernels: momentum with the per-matrix Frobenius norm (double-float
// accumulation, fixed-order fp64 reduction), the bf16 normalisation, and the
// update of master and bf16 copy. Readings (the pages give no coefficients):
// Nesterov momentum M = mu M + g, U = g + mu M; X0 = bf16(U * fp32(1/(|U|+eps)));
// (a, b, c) = (3.4445, -4.7750, 2.0315); wide matrices A = X X^T,
// X = a X + B X; tall ones A = X^T X, X = a X + X B; p = p (1 - lr wd) -
// fp32(lr sqrt(max(1, R/C))) O; the fp32 ops rounded once (-fmad=false).
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <cmath>
#include <cstring>
#include <map>
#include <mutex>
#include <string>
#include <tuple>
#include <vector>

#include "bounds.cuh"
#include "vsf_internal.h"

namespace vsf {
namespace {

constexpr int kMuonThreads = 256;
constexpr int kMuonTargetCtas = 152 * 8;         // fills every SM of the GPU
constexpr int kMaxChunk = 192;                    // matrices in one batched chunk
constexpr int64_t kChunkElems = int64_t(1) << 28;  // bf16 elements of X per chunk (512 MB)

#include "mbarrier.cuh"
#include "ns_gemm.cuh"

// Packed-buffer offset of every matrix of one chunk (kernel parameter).
struct MatTable {
  int64_t off[kMaxChunk];
};

struct DFm {
  float hi = 0.0f, lo = 0.0f;
  __device__ __forceinline__ void add_sq(float x) {
    const float p = __fmul_rn(x, x);
    const float s = __fadd_rn(hi, p);
    const float bp = __fsub_rn(s, hi);
    const float err = __fadd_rn(__fsub_rn(hi, __fsub_rn(s, bp)), __fsub_rn(p, bp));
    hi = s;
    lo = __fadd_rn(__fadd_rn(lo, err), __fmaf_rn(x, x, -p));
  }
};

__device__ __forceinline__ float bf16f(uint16_t h) { return __uint_as_float((uint32_t)h << 16); }
__device__ __forceinline__ uint16_t to_bf16(float x) {
  const __nv_bfloat16 b = __float2bfloat16_rn(x);
  return *reinterpret_cast<const uint16_t*>(&b);
}

// Element access of the three element-wise kernels: V = 8 consecutive
// elements per access (16-byte bf16 and 2 x 16-byte fp32 accesses; every
// matrix offset a multiple of 8) or V = 1.
template <int V>
struct Vec;
template <>
struct Vec<1> {
  static __device__ __forceinline__ void load_bf(const uint16_t* p, float* x) { x[0] = bf16f(*p); }
  static __device__ __forceinline__ void load_f(const float* p, float* x) { x[0] = *p; }
  static __device__ __forceinline__ void store_f(float* p, const float* x) { *p = x[0]; }
  static __device__ __forceinline__ void store_bf(uint16_t* p, const float* x) { *p = to_bf16(x[0]); }
};
template <>
struct Vec<8> {
  static __device__ __forceinline__ void load_bf(const uint16_t* p, float* x) {
    const uint4 u = __ldg(reinterpret_cast<const uint4*>(p));
    const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      x[2 * j] = __uint_as_float(w[j] << 16);
      x[2 * j + 1] = __uint_as_float(w[j] & 0xFFFF0000u);
    }
  }
  static __device__ __forceinline__ void load_f(const float* p, float* x) {
    const float4 a = *reinterpret_cast<const float4*>(p);
    const float4 b = *reinterpret_cast<const float4*>(p + 4);
    x[0] = a.x; x[1] = a.y; x[2] = a.z; x[3] = a.w;
    x[4] = b.x; x[5] = b.y; x[6] = b.z; x[7] = b.w;
  }
  static __device__ __forceinline__ void store_f(float* p, const float* x) {
    *reinterpret_cast<float4*>(p) = make_float4(x[0], x[1], x[2], x[3]);
    *reinterpret_cast<float4*>(p + 4) = make_float4(x[4], x[5], x[6], x[7]);
  }
  static __device__ __forceinline__ void store_bf(uint16_t* p, const float* x) {
    uint32_t w[4];
#pragma unroll
    for (int j = 0; j < 4; ++j)
      w[j] = (uint32_t)to_bf16(x[2 * j]) | ((uint32_t)to_bf16(x[2 * j + 1]) << 16);
    *reinterpret_cast<uint4*>(p) = make_uint4(w[0], w[1], w[2], w[3]);
  }
};

// grid (per, batch): M = mu M + g; partial sums of U^2, U = g + mu M, one
// per CTA of each matrix (partials[j * per + x]).
template <int V>
__global__ void __launch_bounds__(kMuonThreads) muon_momentum_kernel(
    const uint16_t* __restrict__ g, float* M, const __grid_constant__ MatTable tab, int64_t mat,
    float mu, double* partials, Bounds bd) {
  const int64_t off = tab.off[blockIdx.y];
  if (!in_bounds(bd, off, off + mat)) return;  // the whole CTA: uniform
  DFm acc;
  for (int64_t i = ((int64_t)blockIdx.x * kMuonThreads + threadIdx.x) * V; i < mat;
       i += (int64_t)gridDim.x * kMuonThreads * V) {
    float gi[V], m[V];
    Vec<V>::load_bf(g + off + i, gi);
    Vec<V>::load_f(M + off + i, m);
#pragma unroll
    for (int j = 0; j < V; ++j) {
      m[j] = __fadd_rn(__fmul_rn(mu, m[j]), gi[j]);
      acc.add_sq(__fadd_rn(gi[j], __fmul_rn(mu, m[j])));
    }
    Vec<V>::store_f(M + off + i, m);
  }
  __shared__ double red[kMuonThreads / 32];
  double v = isinf(acc.hi) ? (double)acc.hi : (double)acc.hi + (double)acc.lo;
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = v;
  __syncthreads();
  if (threadIdx.x == 0) {
    double s = 0.0;
    for (int w = 0; w < kMuonThreads / 32; ++w) s += red[w];
    partials[(int64_t)blockIdx.y * gridDim.x + blockIdx.x] = s;
  }
}

// X0 = bf16(U * r), U = g + mu M (the momentum already updated), r =
// fp32(1 / (sqrt(sum of the matrix's partials) + eps)); every CTA of a matrix
// reduces the same partials in the same fixed order, so all agree on r. X
// holds the chunk's matrices back to back.
template <int V>
__global__ void __launch_bounds__(kMuonThreads) muon_normalize_kernel(
    const uint16_t* __restrict__ g, const float* __restrict__ M, const __grid_constant__ MatTable tab,
    int64_t mat, float mu, const double* __restrict__ partials, double eps, uint16_t* X,
    Bounds bd) {
  if (!in_bounds(bd, tab.off[blockIdx.y], tab.off[blockIdx.y] + mat)) return;  // uniform
  __shared__ double red[kMuonThreads / 32];
  __shared__ float r_s;
  {
    const double* p = partials + (int64_t)blockIdx.y * gridDim.x;
    double v = 0.0;
    for (unsigned i = threadIdx.x; i < gridDim.x; i += kMuonThreads) v += p[i];
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = v;
    __syncthreads();
    if (threadIdx.x == 0) {
      double s = 0.0;
      for (int w = 0; w < kMuonThreads / 32; ++w) s += red[w];
      r_s = __double2float_rn(1.0 / (sqrt(s) + eps));
    }
    __syncthreads();
  }
  const float re = r_s;
  const int64_t off = tab.off[blockIdx.y];
  uint16_t* x = X + (int64_t)blockIdx.y * mat;
  for (int64_t i = ((int64_t)blockIdx.x * kMuonThreads + threadIdx.x) * V; i < mat;
       i += (int64_t)gridDim.x * kMuonThreads * V) {
    float gi[V], m[V], u[V];
    Vec<V>::load_bf(g + off + i, gi);
    Vec<V>::load_f(M + off + i, m);
#pragma unroll
    for (int j = 0; j < V; ++j) u[j] = __fmul_rn(__fadd_rn(gi[j], __fmul_rn(mu, m[j])), re);
    Vec<V>::store_bf(x + i, u);
  }
}

// p = p * decay - alpha * O; bf16 copy.
template <int V>
__global__ void __launch_bounds__(kMuonThreads) muon_update_kernel(
    const uint16_t* __restrict__ O, float* master, uint16_t* bf, const __grid_constant__ MatTable tab,
    int64_t mat, float decay, float alpha, Bounds bd) {
  const int64_t off = tab.off[blockIdx.y];
  if (!in_bounds(bd, off, off + mat)) return;
  const uint16_t* o = O + (int64_t)blockIdx.y * mat;
  for (int64_t i = ((int64_t)blockIdx.x * kMuonThreads + threadIdx.x) * V; i < mat;
       i += (int64_t)gridDim.x * kMuonThreads * V) {
    float ov[V], p[V];
    Vec<V>::load_bf(o + i, ov);
    Vec<V>::load_f(master + off + i, p);
#pragma unroll
    for (int j = 0; j < V; ++j) p[j] = __fsub_rn(__fmul_rn(p[j], decay), __fmul_rn(alpha, ov[j]));
    Vec<V>::store_f(master + off + i, p);
    Vec<V>::store_bf(bf + off + i, p);
  }
}

struct MuonMatrix {
  int tensor;
  int64_t batch, R, C;
};

std::vector<MuonMatrix> muon_matrices(const vsf_plan* plan) {
  std::vector<MuonMatrix> out;
  for (int t = 0; t < plan->n; ++t) {
    const TensorInfo& x = plan->tensors[t];
    if (x.ndim < 2) continue;
    MuonMatrix mm;
    mm.tensor = t;
    mm.R = x.shape[x.ndim - 2];
    mm.C = x.shape[x.ndim - 1];
    mm.batch = x.numel / (mm.R * mm.C);
    out.push_back(mm);
  }
  return out;
}

double ns_flops(const MuonMatrix& mm) {
  const double n = (double)std::min(mm.R, mm.C), k = (double)std::max(mm.R, mm.C);
  return (double)mm.batch * (4.0 * n * n * k + 2.0 * n * n * n);
}

// Matrices of one shape, batched through the same launches: every matrix of
// every tensor of that shape, in tensor order, cut into chunks of at most
// kMaxChunk matrices and kChunkElems elements.
struct MuonChunk {
  int64_t R, C, batch;
  std::vector<int64_t> off;  // packed offset of each matrix
};

std::vector<MuonChunk> muon_chunks(const vsf_plan* plan) {
  std::vector<std::pair<int64_t, int64_t>> shapes;
  std::vector<std::vector<int64_t>> offs;
  for (const MuonMatrix& mm : muon_matrices(plan)) {
    size_t s = 0;
    while (s < shapes.size() && shapes[s] != std::make_pair(mm.R, mm.C)) ++s;
    if (s == shapes.size()) {
      shapes.push_back({mm.R, mm.C});
      offs.emplace_back();
    }
    const int64_t base = plan->tensors[mm.tensor].offset;
    for (int64_t e = 0; e < mm.batch; ++e) offs[s].push_back(base + e * mm.R * mm.C);
  }
  std::vector<MuonChunk> out;
  for (size_t s = 0; s < shapes.size(); ++s) {
    const int64_t mat = shapes[s].first * shapes[s].second;
    const int64_t cap = std::max<int64_t>(1, std::min<int64_t>(kMaxChunk, kChunkElems / mat));
    for (size_t i = 0; i < offs[s].size(); i += (size_t)cap) {
      MuonChunk c;
      c.R = shapes[s].first;
      c.C = shapes[s].second;
      const size_t end = std::min(offs[s].size(), i + (size_t)cap);
      c.off.assign(offs[s].begin() + i, offs[s].begin() + end);
      c.batch = (int64_t)c.off.size();
      out.push_back(std::move(c));
    }
  }
  return out;
}

// CTAs per matrix for the element-wise kernels: enough to fill the GPU,
// at least 4 elements per thread.
int muon_per(int64_t batch, int64_t mat) {
  const int64_t want = (kMuonTargetCtas + batch - 1) / batch;
  const int64_t most = std::max<int64_t>(1, mat / (8 * kMuonThreads));
  return (int)std::max<int64_t>(1, std::min(want, most));
}

// The chunks run on kMuonLanes stream lanes: lane 0 on the caller's stream,
// the others on the plan's own streams, forked from and joined back into the
// caller's stream. The chunks of different shapes are independent, so one
// lane's launches fill the SMs that another's last partial round of tiles
// (and its element-wise kernels) leave idle. Chunks go to the lane with the
// fewest Newton-Schulz FLOPs so far, largest first, and keep their order
// within a lane; each lane has its own workspace. Measured Muon steps (same
// box): four lanes against two took 2% off the MoE layer (4 batches) and the
// 1.3B model (8), and moved the Llama layer (3) and DSv3 block (2) within 1%;
// two lanes against one took 2-7% off every workload.
#ifndef VSF_MUON_LANES
#define VSF_MUON_LANES 4
#endif
constexpr int kMuonLanes = VSF_MUON_LANES;
static_assert(kMuonLanes >= 1 && kMuonLanes <= 8, "1 to 8 stream lanes");

std::vector<int> muon_lane_of(const std::vector<MuonChunk>& chunks) {
  std::vector<int> order(chunks.size()), lane(chunks.size(), 0);
  std::vector<double> fl(chunks.size());
  for (size_t i = 0; i < chunks.size(); ++i) {
    order[i] = (int)i;
    MuonMatrix mm;
    mm.tensor = 0;
    mm.batch = chunks[i].batch;
    mm.R = chunks[i].R;
    mm.C = chunks[i].C;
    fl[i] = ns_flops(mm);
  }
  std::stable_sort(order.begin(), order.end(), [&](int a, int b) { return fl[a] > fl[b]; });
  double load[kMuonLanes] = {};
  for (int i : order) {
    int l = 0;
    for (int j = 1; j < kMuonLanes; ++j)
      if (load[j] < load[l]) l = j;
    lane[(size_t)i] = l;
    load[l] += fl[(size_t)i];
  }
  return lane;
}

struct MuonLaneLayout {
  size_t partials = 0, x = 0, xn = 0, a = 0, b = 0;
};
struct MuonLayout {
  MuonLaneLayout lane[kMuonLanes];
  size_t bytes = 0;
};

MuonLayout muon_layout(const vsf_plan* plan) {
  const std::vector<MuonChunk> chunks = muon_chunks(plan);
  const std::vector<int> lane_of = muon_lane_of(chunks);
  int64_t max_elems[kMuonLanes] = {}, max_sq[kMuonLanes] = {}, max_part[kMuonLanes] = {};
  for (size_t i = 0; i < chunks.size(); ++i) {
    const MuonChunk& c = chunks[i];
    const int l = lane_of[i];
    const int64_t n = std::min(c.R, c.C);
    max_elems[l] = std::max(max_elems[l], c.batch * c.R * c.C);
    max_sq[l] = std::max(max_sq[l], c.batch * n * n);
    max_part[l] = std::max(max_part[l], c.batch * muon_per(c.batch, c.R * c.C));
  }
  MuonLayout L;
  size_t cur = 0;
  auto section = [&](size_t bytes) {
    size_t at = (cur + 255) / 256 * 256;
    cur = at + bytes;
    return at;
  };
  for (int l = 0; l < kMuonLanes; ++l) {
    L.lane[l].partials = section(sizeof(double) * std::max<int64_t>(1, max_part[l]));
    L.lane[l].x = section(2 * std::max<int64_t>(1, max_elems[l]));
    L.lane[l].xn = section(2 * std::max<int64_t>(1, max_elems[l]));
    L.lane[l].a = section(2 * std::max<int64_t>(1, max_sq[l]));
    L.lane[l].b = section(2 * std::max<int64_t>(1, max_sq[l]));
  }
  L.bytes = (cur + 255) / 256 * 256;
  return L;
}

// The plan's lanes beyond the caller's stream: a non-blocking stream and a
// join event each, and the fork event.
struct MuonLanes {
  int device = -1;
  cudaStream_t stream[kMuonLanes] = {};  // [0] unused: the caller's stream
  cudaEvent_t join[kMuonLanes] = {};
  cudaEvent_t fork = nullptr;
};

void muon_lanes_free(void* p) {
  MuonLanes* ml = static_cast<MuonLanes*>(p);
  if (ml == nullptr) return;
  if (ml->fork) cudaEventDestroy(ml->fork);
  for (int l = 1; l < kMuonLanes; ++l) {
    if (ml->join[l]) cudaEventDestroy(ml->join[l]);
    if (ml->stream[l]) cudaStreamDestroy(ml->stream[l]);
  }
  delete ml;
}

// cuTensorMapEncodeTiled through the runtime's driver entry point (no link
// against libcuda).
PFN_cuTensorMapEncodeTiled_v12000 gemm_map_encoder() {
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

// Tensor map of one GEMM operand over a strided batch of row-major bf16
// matrices (leading dimension ld, batch stride bs, in elements). K-major:
// `rows` rows of K elements, box 64 K x box_rows rows. MN-major: K rows of
// `rows` (the M or N extent) elements, box 64 x 64. 128-byte swizzle; copies
// outside the matrix read zeros.
vsf_status gemm_operand_map(CUtensorMap* map, const uint16_t* ptr, bool mn, int64_t rows,
                            int64_t K, int64_t ld, int64_t bs, int64_t batch, int box_rows) {
  PFN_cuTensorMapEncodeTiled_v12000 encode = gemm_map_encoder();
  if (encode == nullptr) return fail(VSF_ERR_CUDA, "cuTensorMapEncodeTiled is unavailable");
  cuuint64_t dims[3] = {(cuuint64_t)(mn ? rows : K), (cuuint64_t)(mn ? K : rows),
                        (cuuint64_t)batch};
  cuuint64_t strides[2] = {(cuuint64_t)ld * 2, (cuuint64_t)std::max<int64_t>(bs, ld) * 2};
  cuuint32_t box[3] = {64, (cuuint32_t)(mn ? 64 : box_rows), 1};
  cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = encode(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<uint16_t*>(ptr), dims,
                      strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                      CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                      CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS)
    return fail(VSF_ERR_CUDA, "cuTensorMapEncodeTiled failed (" + std::to_string((int)r) + ")");
  return VSF_OK;
}

template <bool AMN, bool BMN, bool SYM>
vsf_status launch_ns_gemm(const CUtensorMap& ma, const CUtensorMap& mb, const NsGemmArgs& g,
                          unsigned* err, cudaStream_t st) {
  constexpr int CL = 2;  // the CTA pair of one 256 x 256 tile
  constexpr uint32_t kSmem = kGemmSmem;
  auto fn = ns_gemm_kernel<AMN, BMN, SYM>;
  // per instantiation and device, once: the shared memory limit and how many
  // clusters fit on the GPU at a time (the persistent grid's size)
  int dev = 0;
  cudaError_t de = cudaGetDevice(&dev);
  if (de != cudaSuccess || dev < 0 || dev >= 64)
    return fail(VSF_ERR_CUDA, std::string("ns_gemm: device ") +
                                  (de != cudaSuccess ? cudaGetErrorString(de) : "id out of range"));
  static std::mutex mu;
  static int cached[64] = {};  // 0: not looked up yet
  std::lock_guard<std::mutex> lock(mu);
  int& max_clusters = cached[dev];
  if (max_clusters == 0) max_clusters = [&] {
    if (cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSmem) !=
        cudaSuccess)
      return -1;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(CL * 64);
    cfg.blockDim = dim3(kGemmThreads);
    cfg.dynamicSmemBytes = kSmem;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = CL;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    int n = 0;
    if (cudaOccupancyMaxActiveClusters(&n, fn, &cfg) != cudaSuccess) return -1;
    return std::max(1, n);
  }();
  if (max_clusters < 1) {
    max_clusters = 0;  // look up again next time
    const cudaError_t e = cudaGetLastError();
    return fail(VSF_ERR_CUDA, std::string("ns_gemm (set-up): ") + cudaGetErrorString(e));
  }
  const int items = g.batch * g.tiles_per_matrix;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)(CL * std::max(1, std::min(max_clusters, items))));
  cfg.blockDim = dim3(kGemmThreads);
  cfg.dynamicSmemBytes = kSmem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = CL;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  const cudaError_t e = cudaLaunchKernelEx(&cfg, fn, ma, mb, g, err);
  return e == cudaSuccess ? VSF_OK : fail(VSF_ERR_CUDA, std::string("ns_gemm: ") + cudaGetErrorString(e));
}

template <bool AMN, bool BMN, bool SYM>
vsf_status launch_ns_gemm_simt(const uint16_t* A, int64_t lda, int64_t sa, const uint16_t* B,
                               int64_t ldb, int64_t sb, const NsGemmArgs& g, cudaStream_t st) {
  const dim3 grid((unsigned)((g.N + 15) / 16), (unsigned)((g.M + 15) / 16), (unsigned)g.batch);
  ns_gemm_simt_kernel<AMN, BMN, SYM><<<grid, 256, 0, st>>>(A, lda, sa, B, ldb, sb, g);
  const cudaError_t e = cudaGetLastError();
  return e == cudaSuccess ? VSF_OK : fail(VSF_ERR_CUDA, std::string("ns_gemm: ") + cudaGetErrorString(e));
}

bool tma_ok(const void* p, int64_t ld, int64_t bs) {
  return (reinterpret_cast<uintptr_t>(p) & 15) == 0 && ld % 8 == 0 && bs % 8 == 0;
}

// D[b] = alpha * opA[b] opB[b]^T + beta * C[b] over a strided batch (see
// ns_gemm.cuh). Operand combinations: K-major x K-major (symmetric or not),
// MN-major x MN-major (symmetric), K-major x MN-major. The tensor-core
// kernel needs leading dimensions and batch strides that are multiples of 8
// elements and 16-byte aligned operands; anything else takes the CUDA-core
// kernel.
vsf_status ns_gemm(bool a_mn, bool b_mn, bool sym, int64_t M, int64_t N, int64_t K, int64_t batch,
                   const uint16_t* A, int64_t lda, int64_t sa, const uint16_t* B, int64_t ldb,
                   int64_t sb, float alpha, float beta, const uint16_t* C, int64_t ldc, int64_t sc,
                   uint16_t* D, int64_t ldd, int64_t sd, unsigned* err, cudaStream_t st) {
  if (M < 1 || N < 1 || K < 1 || batch < 1 || M > INT32_MAX || N > INT32_MAX || K > INT32_MAX ||
      batch > 65535)
    return fail(VSF_ERR_ARG, "ns_gemm: sizes out of range");
  if (sym && (M != N || a_mn != b_mn)) return fail(VSF_ERR_ARG, "ns_gemm: symmetric needs opA = opB");
  NsGemmArgs g{};
  g.M = (int)M;
  g.N = (int)N;
  g.K = (int)K;
  g.batch = (int)batch;
  g.alpha = alpha;
  g.beta = beta;
  g.C = C;
  g.ldc = ldc;
  g.sc = sc;
  g.D = D;
  g.ldd = ldd;
  g.sd = sd;
  const int nblocks = (int)((N + kGemmBN - 1) / kGemmBN);
  {
    // work items of the tensor-core kernel: 256 x 256 output tiles (one per
    // CTA pair); a symmetric product keeps in column block J the 256-row
    // groups 0 .. J
    const int64_t rows = 2 * (int64_t)kGemmBM;
    g.mgroups = (int)((M + rows - 1) / rows);
    int64_t items = 0;
    for (int J = 0; J < nblocks; ++J)
      items += sym ? std::min<int64_t>(g.mgroups, J + 1) : g.mgroups;
    if (items * batch >= INT32_MAX) return fail(VSF_ERR_ARG, "ns_gemm: too many tiles");
    g.tiles_per_matrix = (int)items;
  }
  const bool tc = tma_ok(A, lda, sa) && tma_ok(B, ldb, sb) && tma_ok(D, ldd, sd) &&
                  (beta == 0.0f || tma_ok(C, ldc, sc));
  if (!tc) {
    if (!a_mn && !b_mn && sym) return launch_ns_gemm_simt<false, false, true>(A, lda, sa, B, ldb, sb, g, st);
    if (!a_mn && !b_mn) return launch_ns_gemm_simt<false, false, false>(A, lda, sa, B, ldb, sb, g, st);
    if (a_mn && b_mn && sym) return launch_ns_gemm_simt<true, true, true>(A, lda, sa, B, ldb, sb, g, st);
    if (!a_mn && b_mn && !sym) return launch_ns_gemm_simt<false, true, false>(A, lda, sa, B, ldb, sb, g, st);
    return fail(VSF_ERR_ARG, "ns_gemm: unsupported operand layout");
  }
  CUtensorMap ma, mb;
  vsf_status s = gemm_operand_map(&ma, A, a_mn, M, K, lda, sa, batch, kGemmBM);
  // a cluster pair loads half of each opB slice per CTA
  // each CTA of the pair loads its own 128 rows of opA and of opB
  if (s == VSF_OK) s = gemm_operand_map(&mb, B, b_mn, N, K, ldb, sb, batch, kGemmBN / 2);
  if (s != VSF_OK) return s;
  if (!a_mn && !b_mn && sym) return launch_ns_gemm<false, false, true>(ma, mb, g, err, st);
  if (!a_mn && !b_mn) return launch_ns_gemm<false, false, false>(ma, mb, g, err, st);
  if (a_mn && b_mn && sym) return launch_ns_gemm<true, true, true>(ma, mb, g, err, st);
  if (!a_mn && b_mn && !sym) return launch_ns_gemm<false, true, false>(ma, mb, g, err, st);
  return fail(VSF_ERR_ARG, "ns_gemm: unsupported operand layout");
}

}  // namespace

vsf_status muon_lanes_create(vsf_plan* plan) {
  MuonLanes* have = static_cast<MuonLanes*>(plan->muon_lanes);
  if (have != nullptr && have->device == plan->device) return VSF_OK;
  if (plan->muon_lanes_free != nullptr) plan->muon_lanes_free(plan->muon_lanes);
  plan->muon_lanes = nullptr;
  plan->muon_lanes_free = nullptr;
  MuonLanes* ml = new MuonLanes();
  ml->device = plan->device;
  cudaError_t e = cudaEventCreateWithFlags(&ml->fork, cudaEventDisableTiming);
  for (int l = 1; l < kMuonLanes && e == cudaSuccess; ++l) {
    e = cudaStreamCreateWithFlags(&ml->stream[l], cudaStreamNonBlocking);
    if (e == cudaSuccess) e = cudaEventCreateWithFlags(&ml->join[l], cudaEventDisableTiming);
  }
  if (e != cudaSuccess) {
    muon_lanes_free(ml);
    return fail(VSF_ERR_CUDA, std::string("vsf_plan_upload (Muon stream): ") + cudaGetErrorString(e));
  }
  plan->muon_lanes = ml;
  plan->muon_lanes_free = muon_lanes_free;
  return VSF_OK;
}

}  // namespace vsf

using namespace vsf;

extern "C" {

vsf_status vsf_ns_gemm(int32_t a_mn, int32_t b_mn, int32_t sym, int64_t M, int64_t N, int64_t K,
                       int64_t batch, const uint16_t* A, int64_t lda, int64_t sa, const uint16_t* B,
                       int64_t ldb, int64_t sb, float alpha, float beta, const uint16_t* C,
                       int64_t ldc, int64_t sc, uint16_t* D, int64_t ldd, int64_t sd,
                       unsigned* d_err, void* stream) {
  vsf::Range nvtx_range("vsf_ns_gemm");
  if (A == nullptr || B == nullptr || D == nullptr || d_err == nullptr ||
      (beta != 0.0f && C == nullptr))
    return fail(VSF_ERR_ARG, "vsf_ns_gemm: NULL argument");
  if (lda < 1 || ldb < 1 || ldd < 1 || (beta != 0.0f && ldc < 1) || sa < 0 || sb < 0 || sd < 0 ||
      sc < 0)
    return fail(VSF_ERR_ARG, "vsf_ns_gemm: bad leading dimension or batch stride");
  if (!((a_mn == 0 && b_mn == 0) || (a_mn && b_mn && sym) || (a_mn == 0 && b_mn && !sym)))
    return fail(VSF_ERR_ARG, "vsf_ns_gemm: operand layouts must be K/K, MN/MN (symmetric) or K/MN");
  return ns_gemm(a_mn != 0, b_mn != 0, sym != 0, M, N, K, batch, A, lda, sa, B, ldb, sb, alpha,
                 beta, C, ldc, sc, D, ldd, sd, d_err, static_cast<cudaStream_t>(stream));
}

vsf_status vsf_muon_select_roots(const vsf_plan* plan, int32_t* root, double* load_balance) {
  if (plan == nullptr || root == nullptr) return fail(VSF_ERR_ARG, "vsf_muon_select_roots: NULL");
  std::vector<MuonMatrix> mats = muon_matrices(plan);
  std::vector<int> order(mats.size());
  for (size_t i = 0; i < order.size(); ++i) order[i] = (int)i;
  std::stable_sort(order.begin(), order.end(),
                   [&](int a, int b) { return ns_flops(mats[a]) > ns_flops(mats[b]); });
  std::vector<double> load(plan->m, 0.0);
  for (int t = 0; t < plan->n; ++t) root[t] = -1;
  for (int i : order) {
    int best = 0;
    for (int r = 1; r < plan->m; ++r)
      if (load[r] < load[best]) best = r;
    root[mats[i].tensor] = best;
    load[best] += ns_flops(mats[i]);
  }
  if (load_balance) {
    double mx = 0.0, sum = 0.0;
    for (double l : load) {
      mx = std::max(mx, l);
      sum += l;
    }
    *load_balance = sum > 0.0 ? mx / (sum / plan->m) : 1.0;
  }
  return VSF_OK;
}

size_t vsf_muon_workspace_bytes(const vsf_plan* plan) {
  return plan == nullptr ? 0 : muon_layout(plan).bytes;
}

int32_t vsf_muon_chunk_count(const vsf_plan* plan) {
  return plan == nullptr ? 0 : (int32_t)muon_chunks(plan).size();
}

int64_t vsf_muon_kernel_launches(const vsf_plan* plan, int32_t ns_steps) {
  if (plan == nullptr || ns_steps < 0) return 0;
  int64_t n = 0;
  for (const MuonChunk& c : muon_chunks(plan)) {
    const int64_t nm = std::min(c.R, c.C);
    (void)nm;
    n += 3 + 3 * (int64_t)ns_steps;  // momentum, normalise, update; 3 products per iteration
  }
  return n;
}

vsf_status vsf_muon_step(const vsf_plan* plan, const uint16_t* packed_grad, float* momentum,
                         float* master, uint16_t* packed_bf16, const vsf_muon_hparams* hp,
                         void* d_workspace, size_t ws_bytes, void* stream) {
  vsf::Range nvtx_range("vsf_muon_step");
  if (plan == nullptr || packed_grad == nullptr || momentum == nullptr || master == nullptr ||
      packed_bf16 == nullptr || hp == nullptr || d_workspace == nullptr)
    return fail(VSF_ERR_ARG, "vsf_muon_step: NULL argument");
  if (!plan->uploaded) return fail(VSF_ERR_STATE, "vsf_muon_step: plan not uploaded");
  if (plan->rank_begin != 0 || plan->rank_end != plan->m)
    return fail(VSF_ERR_STATE, "vsf_muon_step: Newton-Schulz needs whole matrices (unrestricted plan)");
  const MuonLayout L = muon_layout(plan);
  if (ws_bytes < L.bytes) return fail(VSF_ERR_ARG, "vsf_muon_step: workspace too small");
  for (const void* p : {(const void*)packed_grad, (const void*)momentum, (const void*)master,
                        (const void*)packed_bf16, (const void*)d_workspace})
    if (reinterpret_cast<uintptr_t>(p) & 15)
      return fail(VSF_ERR_ALIGN, "vsf_muon_step: pointer not 16-byte aligned");
  if (hp->ns_steps < 0) return fail(VSF_ERR_ARG, "vsf_muon_step: ns_steps must be >= 0");
  const MuonLanes* ml = static_cast<const MuonLanes*>(plan->muon_lanes);
  if (ml == nullptr) return fail(VSF_ERR_STATE, "vsf_muon_step: plan has no Muon stream");
  const std::vector<MuonChunk> chunks = muon_chunks(plan);
  const std::vector<int> lane_of = muon_lane_of(chunks);
  bool used[kMuonLanes] = {};
  for (int l : lane_of) used[l] = true;
  cudaStream_t caller = static_cast<cudaStream_t>(stream);
  cudaStream_t lanes[kMuonLanes];
  bool forked = false;
  for (int l = 0; l < kMuonLanes; ++l) {
    lanes[l] = l == 0 ? caller : ml->stream[l];
    forked = forked || (l > 0 && used[l]);
  }
  unsigned char* ws = static_cast<unsigned char*>(d_workspace);
  unsigned* err = reinterpret_cast<unsigned*>(plan->d_ws + plan->layout.error);
  const float mu = (float)hp->momentum;
  const float decay = (float)(1.0 - hp->lr * hp->weight_decay);
  const float na = (float)hp->ns_a, nb = (float)hp->ns_b, nc = (float)hp->ns_c;
  const Bounds bd{plan->total, reinterpret_cast<unsigned*>(plan->d_ws + plan->layout.error)};

  if (forked) {  // the other lanes start after the caller's earlier work
    cudaError_t e = cudaEventRecord(ml->fork, caller);
    for (int l = 1; l < kMuonLanes && e == cudaSuccess; ++l)
      if (used[l]) e = cudaStreamWaitEvent(lanes[l], ml->fork, 0);
    if (e != cudaSuccess)
      return fail(VSF_ERR_CUDA, std::string("vsf_muon_step (fork): ") + cudaGetErrorString(e));
  }
  // Enqueues every chunk of the step; the caller's stream then waits for the
  // other lanes, also when an enqueue failed part way.
  auto run = [&]() -> vsf_status {
    for (size_t ci = 0; ci < chunks.size(); ++ci) {
      const MuonChunk& c = chunks[ci];
      const int lane = lane_of[ci];
      cudaStream_t st = lanes[lane];
      const MuonLaneLayout& LL = L.lane[lane];
      double* partials = reinterpret_cast<double*>(ws + LL.partials);
      uint16_t* X = reinterpret_cast<uint16_t*>(ws + LL.x);
      uint16_t* Xn = reinterpret_cast<uint16_t*>(ws + LL.xn);
      uint16_t* A = reinterpret_cast<uint16_t*>(ws + LL.a);
      uint16_t* B = reinterpret_cast<uint16_t*>(ws + LL.b);
      MatTable tab;
      for (int64_t j = 0; j < c.batch; ++j) tab.off[j] = c.off[(size_t)j];
      const int64_t mat = c.R * c.C;
      const int per = muon_per(c.batch, mat);
      const dim3 grid((unsigned)per, (unsigned)c.batch);
      // 8-wide accesses when every matrix of the chunk starts on 8 elements
      bool vec = mat % 8 == 0;
      for (int64_t j = 0; j < c.batch; ++j) vec = vec && c.off[(size_t)j] % 8 == 0;
      if (vec) {
        muon_momentum_kernel<8><<<grid, kMuonThreads, 0, st>>>(packed_grad, momentum, tab, mat, mu,
                                                               partials, bd);
        muon_normalize_kernel<8><<<grid, kMuonThreads, 0, st>>>(packed_grad, momentum, tab, mat, mu,
                                                                partials, hp->eps, X, bd);
      } else {
        muon_momentum_kernel<1><<<grid, kMuonThreads, 0, st>>>(packed_grad, momentum, tab, mat, mu,
                                                               partials, bd);
        muon_normalize_kernel<1><<<grid, kMuonThreads, 0, st>>>(packed_grad, momentum, tab, mat, mu,
                                                                partials, hp->eps, X, bd);
      }
      cudaError_t e = cudaGetLastError();
      if (e != cudaSuccess) return fail(VSF_ERR_CUDA, std::string("vsf_muon_step: ") + cudaGetErrorString(e));
      // Newton-Schulz on the row-major R x C matrices of the chunk (X holds
      // them back to back, stride R*C; A and B are n x n, n = min(R, C)).
      // Wide (R <= C): A = X X^T, B = c A A + b A, X' = a X + B X.
      // Tall (R > C):  A = X^T X, B = c A A + b A, X' = a X + X B.
      // A and B are symmetric, so the B operand of A A is A's rows and that of
      // X B is B's rows; X^T X reads X's columns (MN-major) and B X reads X's
      // columns as its second operand.
      const bool tall = c.R > c.C;
      const int64_t n = std::min(c.R, c.C), k = std::max(c.R, c.C), sx = mat, sa = n * n;
      for (int it = 0; it < hp->ns_steps; ++it) {
        vsf_status s = VSF_OK;
        if (!tall)
          s = ns_gemm(false, false, true, n, n, k, c.batch, X, c.C, sx, X, c.C, sx, 1.0f, 0.0f,
                      nullptr, n, sa, A, n, sa, err, st);
        else
          s = ns_gemm(true, true, true, n, n, k, c.batch, X, c.C, sx, X, c.C, sx, 1.0f, 0.0f,
                      nullptr, n, sa, A, n, sa, err, st);
        if (s == VSF_OK)
          s = ns_gemm(false, false, true, n, n, n, c.batch, A, n, sa, A, n, sa, nc, nb, A, n, sa, B,
                      n, sa, err, st);
        if (s == VSF_OK) {
          if (!tall)  // X'[i][l] = a X[i][l] + sum_j B[i][j] X[j][l]
            s = ns_gemm(false, true, false, n, c.C, n, c.batch, B, n, sa, X, c.C, sx, 1.0f, na, X,
                        c.C, sx, Xn, c.C, sx, err, st);
          else        // X'[l][i] = a X[l][i] + sum_j X[l][j] B[i][j]
            s = ns_gemm(false, false, false, c.R, n, n, c.batch, X, c.C, sx, B, n, sa, 1.0f, na, X,
                        c.C, sx, Xn, c.C, sx, err, st);
        }
        if (s != VSF_OK) return s;
        std::swap(X, Xn);
      }
      const float alpha = (float)(hp->lr * std::sqrt(std::max(1.0, (double)c.R / (double)c.C)));
      if (vec)
        muon_update_kernel<8><<<grid, kMuonThreads, 0, st>>>(X, master, packed_bf16, tab, mat, decay,
                                                             alpha, bd);
      else
        muon_update_kernel<1><<<grid, kMuonThreads, 0, st>>>(X, master, packed_bf16, tab, mat, decay,
                                                             alpha, bd);
      e = cudaGetLastError();
      if (e != cudaSuccess) return fail(VSF_ERR_CUDA, std::string("vsf_muon_step: ") + cudaGetErrorString(e));
    }
    return VSF_OK;
  };
  const vsf_status s = run();
  cudaError_t je = cudaSuccess;  // join: work after the call on the caller's stream sees every lane
  for (int l = 1; l < kMuonLanes; ++l) {
    if (!used[l]) continue;
    cudaError_t e = cudaEventRecord(ml->join[l], lanes[l]);
    if (e == cudaSuccess) e = cudaStreamWaitEvent(caller, ml->join[l], 0);
    if (je == cudaSuccess) je = e;
  }
  if (je != cudaSuccess && s == VSF_OK)
    return fail(VSF_ERR_CUDA, std::string("vsf_muon_step (join): ") + cudaGetErrorString(je));
  return s;
}

}  // extern "C"
