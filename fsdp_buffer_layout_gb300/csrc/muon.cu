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
//                         GEMMs each (cuBLASLt, bf16 operands, fp32
//                         accumulation), batched over a tensor's matrices;
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
#include <cublasLt.h>
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
constexpr size_t kLtWorkspace = 64u << 20;         // cuBLASLt workspace bytes
constexpr int64_t kSymBlockMin = 1024;             // n from which symmetric products use blocks
#ifndef VSF_SYM_LEVELS
#define VSF_SYM_LEVELS 2
#endif
constexpr int kSymLevels = VSF_SYM_LEVELS;         // levels of splitting (a lower one needs 2048)

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

// Symmetric products computed by blocks: an off-diagonal block below the
// diagonal is the transpose of its mirror above it. A is row-major n x n;
// block sizes and offsets are multiples of 8 (rows start on 16 bytes).
// One launch mirrors every block of one product: the grid's x index runs
// over the 64 x 64 tiles of all blocks in turn (tile_begin holds each block's
// first tile), y over the matrices of the chunk. One CTA (8 warps) per tile:
// rows of the source tile are read as 32-bit bf16 pairs (coalesced), kept in
// shared memory (rows padded to 33 words), and each output word pairs the
// same column of two adjacent source rows; output rows are written as
// 32-bit words (coalesced).
constexpr int kMaxMirrors = 4;
struct MirrorBlocks {
  int64_t bi[kMaxMirrors], bj[kMaxMirrors], size[kMaxMirrors];
  int32_t tile_begin[kMaxMirrors + 1];
  int32_t count;
};

__global__ void __launch_bounds__(256) mirror_kernel(uint16_t* A, int64_t n, const __grid_constant__ MirrorBlocks mb,
                                                     int64_t sa) {
  __shared__ uint32_t tile[64][33];
  int q = 0;
  while (q + 1 < mb.count && (int)blockIdx.x >= mb.tile_begin[q + 1]) ++q;
  const int64_t bi = mb.bi[q], bj = mb.bj[q], h = mb.size[q];
  const int64_t tiles = (h + 63) / 64;
  const int64_t tix = (int64_t)blockIdx.x - mb.tile_begin[q];
  uint16_t* M = A + (int64_t)blockIdx.y * sa;
  // the h x h block at rows bi, columns bj, mirrored to rows bj, columns bi
  const int64_t i0 = tix / tiles * 64, j0 = tix % tiles * 64;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  for (int r = warp; r < 64; r += 8) {
    const int64_t i = i0 + r, j = j0 + 2 * lane;
    uint32_t w = 0;
    if (i < h && j + 1 < h) {
      w = *reinterpret_cast<const uint32_t*>(M + (bi + i) * n + bj + j);
    } else if (i < h && j < h) {
      w = M[(bi + i) * n + bj + j];
    }
    tile[r][lane] = w;
  }
  __syncthreads();
  // destination row bj + j0 + c holds source column j0 + c; its word `lane`
  // holds source rows i0 + 2 lane and i0 + 2 lane + 1
  for (int c = warp; c < 64; c += 8) {
    const int64_t orow = j0 + c, ocol = i0 + 2 * lane;
    if (orow >= h || ocol >= h) continue;
    const uint32_t a = tile[2 * lane][c >> 1], b = tile[2 * lane + 1][c >> 1];
    const uint32_t lo = (c & 1) ? (a >> 16) : (a & 0xffffu);
    const uint32_t hi = (c & 1) ? (b >> 16) : (b & 0xffffu);
    uint16_t* dst = M + (bj + orow) * n + bi + ocol;
    if (ocol + 1 < h)
      *reinterpret_cast<uint32_t*>(dst) = lo | (hi << 16);
    else
      *dst = (uint16_t)lo;
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

struct MuonLayout {
  size_t lt = 0, partials = 0, x = 0, xn = 0, a = 0, b = 0, bytes = 0;
};

MuonLayout muon_layout(const vsf_plan* plan) {
  int64_t max_elems = 0, max_sq = 0, max_part = 0;
  for (const MuonChunk& c : muon_chunks(plan)) {
    const int64_t n = std::min(c.R, c.C);
    max_elems = std::max(max_elems, c.batch * c.R * c.C);
    max_sq = std::max(max_sq, c.batch * n * n);
    max_part = std::max(max_part, c.batch * muon_per(c.batch, c.R * c.C));
  }
  MuonLayout L;
  size_t cur = 0;
  auto section = [&](size_t bytes) {
    size_t at = (cur + 255) / 256 * 256;
    cur = at + bytes;
    return at;
  };
  L.lt = section(kLtWorkspace);
  L.partials = section(sizeof(double) * std::max<int64_t>(1, max_part));
  L.x = section(2 * std::max<int64_t>(1, max_elems));
  L.xn = section(2 * std::max<int64_t>(1, max_elems));
  L.a = section(2 * std::max<int64_t>(1, max_sq));
  L.b = section(2 * std::max<int64_t>(1, max_sq));
  L.bytes = (cur + 255) / 256 * 256;
  return L;
}

// cuBLASLt: one handle per process, plans cached by GEMM shape.
struct LtGemm {
  cublasLtMatmulDesc_t op = nullptr;
  cublasLtMatrixLayout_t la = nullptr, lb = nullptr, lc = nullptr;
  cublasLtMatmulAlgo_t algo;
  bool ok = false;
};

std::mutex g_lt_mu;
cublasLtHandle_t g_lt = nullptr;
std::map<std::tuple<int, int, int64_t, int64_t, int64_t, int64_t, int64_t, int64_t, int64_t,
                    uint32_t, uint32_t, uint32_t>,
         LtGemm>
    g_lt_cache;

// Largest power of two (at most 256) dividing the address of every matrix of
// a strided batch; the algorithm heuristic assumes 256 unless told.
uint32_t batch_alignment(const void* p, int64_t stride_elems) {
  uint64_t v = (uint64_t)reinterpret_cast<uintptr_t>(p) | (uint64_t)(stride_elems * 2) | 256u;
  return (uint32_t)(v & (~v + 1));
}

vsf_status lt_fail(cublasStatus_t s, const char* what) {
  return fail(VSF_ERR_CUDA, std::string(what) + ": cuBLASLt status " + std::to_string((int)s));
}

// Column-major D[M x N] = alpha * op(A)[M x K] * op(B)[K x N] + beta * C, bf16
// in and out, fp32 accumulation, strided batch. lda/ldb/ldc are the
// column-major leading dimensions of the stored A, B, C/D.
vsf_status lt_gemm(bool ta, bool tb, int64_t M, int64_t N, int64_t K, const void* A, int64_t lda,
                   int64_t sa, const void* B, int64_t ldb, int64_t sb, float alpha, float beta,
                   const void* C, void* D, int64_t ldc, int64_t sc, int64_t batch, void* ws,
                   cudaStream_t st) {
  std::lock_guard<std::mutex> lock(g_lt_mu);
  cublasStatus_t s;
  if (g_lt == nullptr) {
    s = cublasLtCreate(&g_lt);
    if (s != CUBLAS_STATUS_SUCCESS) return lt_fail(s, "cublasLtCreate");
  }
  const uint32_t al_a = batch_alignment(A, sa), al_b = batch_alignment(B, sb),
                 al_c = std::min(batch_alignment(C, sc), batch_alignment(D, sc));
  auto key = std::make_tuple((int)ta, (int)tb, M, N, K, lda, ldb, ldc, batch, al_a, al_b, al_c);
  LtGemm& g = g_lt_cache[key];
  if (!g.ok) {
    const cublasOperation_t opa = ta ? CUBLAS_OP_T : CUBLAS_OP_N;
    const cublasOperation_t opb = tb ? CUBLAS_OP_T : CUBLAS_OP_N;
    if ((s = cublasLtMatmulDescCreate(&g.op, CUBLAS_COMPUTE_32F, CUDA_R_32F)) != CUBLAS_STATUS_SUCCESS)
      return lt_fail(s, "cublasLtMatmulDescCreate");
    cublasLtMatmulDescSetAttribute(g.op, CUBLASLT_MATMUL_DESC_TRANSA, &opa, sizeof(opa));
    cublasLtMatmulDescSetAttribute(g.op, CUBLASLT_MATMUL_DESC_TRANSB, &opb, sizeof(opb));
    const uint64_t ar = ta ? K : M, ac = ta ? M : K, br = tb ? N : K, bc = tb ? K : N;
    if ((s = cublasLtMatrixLayoutCreate(&g.la, CUDA_R_16BF, ar, ac, lda)) != CUBLAS_STATUS_SUCCESS ||
        (s = cublasLtMatrixLayoutCreate(&g.lb, CUDA_R_16BF, br, bc, ldb)) != CUBLAS_STATUS_SUCCESS ||
        (s = cublasLtMatrixLayoutCreate(&g.lc, CUDA_R_16BF, M, N, ldc)) != CUBLAS_STATUS_SUCCESS)
      return lt_fail(s, "cublasLtMatrixLayoutCreate");
    const int32_t bcount = (int32_t)batch;
    cublasLtMatrixLayoutSetAttribute(g.la, CUBLASLT_MATRIX_LAYOUT_BATCH_COUNT, &bcount, sizeof(bcount));
    cublasLtMatrixLayoutSetAttribute(g.lb, CUBLASLT_MATRIX_LAYOUT_BATCH_COUNT, &bcount, sizeof(bcount));
    cublasLtMatrixLayoutSetAttribute(g.lc, CUBLASLT_MATRIX_LAYOUT_BATCH_COUNT, &bcount, sizeof(bcount));
    cublasLtMatrixLayoutSetAttribute(g.la, CUBLASLT_MATRIX_LAYOUT_STRIDED_BATCH_OFFSET, &sa, sizeof(sa));
    cublasLtMatrixLayoutSetAttribute(g.lb, CUBLASLT_MATRIX_LAYOUT_STRIDED_BATCH_OFFSET, &sb, sizeof(sb));
    cublasLtMatrixLayoutSetAttribute(g.lc, CUBLASLT_MATRIX_LAYOUT_STRIDED_BATCH_OFFSET, &sc, sizeof(sc));
    cublasLtMatmulPreference_t pref;
    cublasLtMatmulPreferenceCreate(&pref);
    const size_t wsb = kLtWorkspace;
    cublasLtMatmulPreferenceSetAttribute(pref, CUBLASLT_MATMUL_PREF_MAX_WORKSPACE_BYTES, &wsb,
                                         sizeof(wsb));
    cublasLtMatmulPreferenceSetAttribute(pref, CUBLASLT_MATMUL_PREF_MIN_ALIGNMENT_A_BYTES, &al_a,
                                         sizeof(al_a));
    cublasLtMatmulPreferenceSetAttribute(pref, CUBLASLT_MATMUL_PREF_MIN_ALIGNMENT_B_BYTES, &al_b,
                                         sizeof(al_b));
    cublasLtMatmulPreferenceSetAttribute(pref, CUBLASLT_MATMUL_PREF_MIN_ALIGNMENT_C_BYTES, &al_c,
                                         sizeof(al_c));
    cublasLtMatmulPreferenceSetAttribute(pref, CUBLASLT_MATMUL_PREF_MIN_ALIGNMENT_D_BYTES, &al_c,
                                         sizeof(al_c));
    cublasLtMatmulHeuristicResult_t res;
    int found = 0;
    s = cublasLtMatmulAlgoGetHeuristic(g_lt, g.op, g.la, g.lb, g.lc, g.lc, pref, 1, &res, &found);
    cublasLtMatmulPreferenceDestroy(pref);
    if (s != CUBLAS_STATUS_SUCCESS || found == 0)
      return lt_fail(s == CUBLAS_STATUS_SUCCESS ? CUBLAS_STATUS_NOT_SUPPORTED : s,
                     "cublasLtMatmulAlgoGetHeuristic");
    g.algo = res.algo;
    g.ok = true;
  }
  s = cublasLtMatmul(g_lt, g.op, &alpha, A, g.la, B, g.lb, &beta, C, g.lc, D, g.lc, &g.algo, ws,
                     kLtWorkspace, st);
  return s == CUBLAS_STATUS_SUCCESS ? VSF_OK : lt_fail(s, "cublasLtMatmul");
}

}  // namespace
}  // namespace vsf

using namespace vsf;

extern "C" {

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
    n += 3 + (nm >= kSymBlockMin && nm % 16 == 0 ? 2 * (int64_t)ns_steps : 0);
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
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  unsigned char* ws = static_cast<unsigned char*>(d_workspace);
  double* partials = reinterpret_cast<double*>(ws + L.partials);
  uint16_t* X = reinterpret_cast<uint16_t*>(ws + L.x);
  uint16_t* Xn = reinterpret_cast<uint16_t*>(ws + L.xn);
  uint16_t* A = reinterpret_cast<uint16_t*>(ws + L.a);
  uint16_t* B = reinterpret_cast<uint16_t*>(ws + L.b);
  void* lt = ws + L.lt;
  const float mu = (float)hp->momentum;
  const float decay = (float)(1.0 - hp->lr * hp->weight_decay);
  const float na = (float)hp->ns_a, nb = (float)hp->ns_b, nc = (float)hp->ns_c;
  const Bounds bd{plan->total, reinterpret_cast<unsigned*>(plan->d_ws + plan->layout.error)};

  for (const MuonChunk& c : muon_chunks(plan)) {
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
    // Newton-Schulz, column-major view of the row-major R x C matrices: Xc is
    // C x R with leading dimension C.
    const bool tall = c.R > c.C;
    const int64_t n = std::min(c.R, c.C), sx = mat, sa = n * n;
    // The two symmetric products (the Gram matrix and c A A + b A) by blocks:
    // a diagonal block of size s >= 1024 (2048 below the top level) splits
    // into two diagonal halves and their off-diagonal block, whose mirror is
    // its transpose. One level costs 3/4 of the FLOPs, two levels 5/8; the
    // results are exactly symmetric. Column-major operand views of the
    // row-major buffers.
    struct Blk {
      int64_t i0, j0, size;
    };
    std::vector<Blk> gemm_blocks, mirrors;
    {
      std::vector<std::pair<Blk, int>> todo = {{{0, 0, n}, 0}};
      while (!todo.empty()) {
        const Blk b = todo.back().first;
        const int level = todo.back().second;
        todo.pop_back();
        const int64_t smin = level == 0 ? kSymBlockMin : 2 * kSymBlockMin;
        if (level < kSymLevels && b.size >= smin && b.size % 16 == 0) {
          const int64_t h2 = b.size / 2;
          todo.push_back({{b.i0, b.i0, h2}, level + 1});
          todo.push_back({{b.i0 + h2, b.i0 + h2, h2}, level + 1});
          gemm_blocks.push_back({b.i0, b.i0 + h2, h2});
          mirrors.push_back({b.i0, b.i0 + h2, h2});
        } else {
          gemm_blocks.push_back(b);
        }
      }
    }
    if (mirrors.size() > (size_t)kMaxMirrors)
      return fail(VSF_ERR_STATE, "vsf_muon_step: too many mirrored blocks");
    MirrorBlocks mb{};
    mb.count = (int32_t)mirrors.size();
    mb.tile_begin[0] = 0;
    for (size_t q = 0; q < mirrors.size(); ++q) {
      mb.bi[q] = mirrors[q].i0;
      mb.bj[q] = mirrors[q].j0;
      mb.size[q] = mirrors[q].size;
      const int64_t t = (mirrors[q].size + 63) / 64;
      mb.tile_begin[q + 1] = mb.tile_begin[q] + (int32_t)(t * t);
    }
    auto mirror_all = [&](uint16_t* M) {
      mirror_kernel<<<dim3((unsigned)mb.tile_begin[mb.count], (unsigned)c.batch), 256, 0, st>>>(
          M, n, mb, sa);
      const cudaError_t e2 = cudaGetLastError();
      return e2 == cudaSuccess ? VSF_OK : fail(VSF_ERR_CUDA, std::string("vsf_muon_step: ") + cudaGetErrorString(e2));
    };
    for (int it = 0; it < hp->ns_steps; ++it) {
      vsf_status s = VSF_OK;
      // A (n x n) = X X^T (wide) or X^T X (tall); block (I, J) at A + I0 n + J0
      for (size_t q = 0; q < gemm_blocks.size() && s == VSF_OK; ++q) {
        const int64_t I0 = gemm_blocks[q].i0, J0 = gemm_blocks[q].j0, hs = gemm_blocks[q].size;
        if (!tall)
          s = lt_gemm(true, false, hs, hs, c.C, X + J0 * c.C, c.C, sx, X + I0 * c.C, c.C, sx, 1.0f,
                      0.0f, A + I0 * n + J0, A + I0 * n + J0, n, sa, c.batch, lt, st);
        else
          s = lt_gemm(false, true, hs, hs, c.R, X + J0, c.C, sx, X + I0, c.C, sx, 1.0f, 0.0f,
                      A + I0 * n + J0, A + I0 * n + J0, n, sa, c.batch, lt, st);
      }
      if (s == VSF_OK && !mirrors.empty()) s = mirror_all(A);
      if (s != VSF_OK) return s;
      // B = c A A + b A (A symmetric: block (I, J) = c A[J rows] A[I cols] + b A_IJ)
      for (size_t q = 0; q < gemm_blocks.size() && s == VSF_OK; ++q) {
        const int64_t I0 = gemm_blocks[q].i0, J0 = gemm_blocks[q].j0, hs = gemm_blocks[q].size;
        s = lt_gemm(false, false, hs, hs, n, A + J0, n, sa, A + I0 * n, n, sa, nc, nb,
                    A + I0 * n + J0, B + I0 * n + J0, n, sa, c.batch, lt, st);
      }
      if (s == VSF_OK && !mirrors.empty()) s = mirror_all(B);
      if (s != VSF_OK) return s;
      // X' = a X + B X (wide) or a X + X B (tall), column-major Xc' = a Xc +
      // Xc B (wide) or a Xc + B Xc (tall)
      if (!tall)
        s = lt_gemm(false, false, c.C, c.R, c.R, X, c.C, sx, B, n, sa, 1.0f, na, X, Xn, c.C, sx,
                    c.batch, lt, st);
      else
        s = lt_gemm(false, false, c.C, c.R, c.C, B, n, sa, X, c.C, sx, 1.0f, na, X, Xn, c.C, sx,
                    c.batch, lt, st);
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
}

}  // extern "C"
