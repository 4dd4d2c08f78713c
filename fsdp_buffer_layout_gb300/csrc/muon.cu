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

#include "vsf_internal.h"

namespace vsf {
namespace {

constexpr int kMuonThreads = 256;
constexpr int kMuonCtasPerMatrix = 64;     // norm partials per matrix
constexpr size_t kLtWorkspace = 64u << 20;  // cuBLASLt workspace bytes

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

// grid (kMuonCtasPerMatrix, nmat): M = mu M + g; partial sums of U^2,
// U = g + mu M, per CTA of each matrix.
__global__ void __launch_bounds__(kMuonThreads) muon_momentum_kernel(
    const uint16_t* __restrict__ g, float* M, int64_t base, int64_t mat, float mu,
    double* partials) {
  const int64_t off = base + (int64_t)blockIdx.y * mat;
  DFm acc;
  for (int64_t i = (int64_t)blockIdx.x * kMuonThreads + threadIdx.x; i < mat;
       i += (int64_t)gridDim.x * kMuonThreads) {
    const float gi = bf16f(g[off + i]);
    const float m = __fadd_rn(__fmul_rn(mu, M[off + i]), gi);
    M[off + i] = m;
    acc.add_sq(__fadd_rn(gi, __fmul_rn(mu, m)));
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

// One thread per matrix: r = fp32(1 / (sqrt(sum) + eps)).
__global__ void muon_scale_kernel(const double* __restrict__ partials, int per, int nmat,
                                  double eps, float* r) {
  const int e = blockIdx.x * blockDim.x + threadIdx.x;
  if (e >= nmat) return;
  double s = 0.0;
  for (int i = 0; i < per; ++i) s += partials[(int64_t)e * per + i];
  r[e] = __double2float_rn(1.0 / (sqrt(s) + eps));
}

// X0 = bf16(U * r), U = g + mu M (the momentum already updated).
__global__ void __launch_bounds__(kMuonThreads) muon_normalize_kernel(
    const uint16_t* __restrict__ g, const float* __restrict__ M, int64_t base, int64_t mat,
    float mu, const float* __restrict__ r, uint16_t* X) {
  const int64_t off = (int64_t)blockIdx.y * mat;
  const float re = r[blockIdx.y];
  for (int64_t i = (int64_t)blockIdx.x * kMuonThreads + threadIdx.x; i < mat;
       i += (int64_t)gridDim.x * kMuonThreads) {
    const float u = __fadd_rn(bf16f(g[base + off + i]), __fmul_rn(mu, M[base + off + i]));
    X[off + i] = to_bf16(__fmul_rn(u, re));
  }
}

// p = p * decay - alpha * O; bf16 copy.
__global__ void __launch_bounds__(kMuonThreads) muon_update_kernel(
    const uint16_t* __restrict__ O, float* master, uint16_t* bf, int64_t base, int64_t n,
    float decay, float alpha) {
  for (int64_t i = (int64_t)blockIdx.x * kMuonThreads + threadIdx.x; i < n;
       i += (int64_t)gridDim.x * kMuonThreads) {
    const float p = __fsub_rn(__fmul_rn(master[base + i], decay), __fmul_rn(alpha, bf16f(O[i])));
    master[base + i] = p;
    bf[base + i] = to_bf16(p);
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

struct MuonLayout {
  size_t lt = 0, partials = 0, r = 0, x = 0, xn = 0, a = 0, b = 0, bytes = 0;
};

MuonLayout muon_layout(const vsf_plan* plan) {
  int64_t max_elems = 0, max_sq = 0, max_batch = 0;
  for (const MuonMatrix& mm : muon_matrices(plan)) {
    const int64_t n = std::min(mm.R, mm.C);
    max_elems = std::max(max_elems, mm.batch * mm.R * mm.C);
    max_sq = std::max(max_sq, mm.batch * n * n);
    max_batch = std::max(max_batch, mm.batch);
  }
  MuonLayout L;
  size_t cur = 0;
  auto section = [&](size_t bytes) {
    size_t at = (cur + 255) / 256 * 256;
    cur = at + bytes;
    return at;
  };
  L.lt = section(kLtWorkspace);
  L.partials = section(sizeof(double) * std::max<int64_t>(1, max_batch) * kMuonCtasPerMatrix);
  L.r = section(sizeof(float) * std::max<int64_t>(1, max_batch));
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

vsf_status vsf_muon_step(const vsf_plan* plan, const uint16_t* packed_grad, float* momentum,
                         float* master, uint16_t* packed_bf16, const vsf_muon_hparams* hp,
                         void* d_workspace, size_t ws_bytes, void* stream) {
  if (plan == nullptr || packed_grad == nullptr || momentum == nullptr || master == nullptr ||
      packed_bf16 == nullptr || hp == nullptr || d_workspace == nullptr)
    return fail(VSF_ERR_ARG, "vsf_muon_step: NULL argument");
  if (!plan->uploaded) return fail(VSF_ERR_STATE, "vsf_muon_step: plan not uploaded");
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
  float* r = reinterpret_cast<float*>(ws + L.r);
  uint16_t* X = reinterpret_cast<uint16_t*>(ws + L.x);
  uint16_t* Xn = reinterpret_cast<uint16_t*>(ws + L.xn);
  uint16_t* A = reinterpret_cast<uint16_t*>(ws + L.a);
  uint16_t* B = reinterpret_cast<uint16_t*>(ws + L.b);
  void* lt = ws + L.lt;
  const float mu = (float)hp->momentum;
  const float decay = (float)(1.0 - hp->lr * hp->weight_decay);
  const float na = (float)hp->ns_a, nb = (float)hp->ns_b, nc = (float)hp->ns_c;

  for (const MuonMatrix& mm : muon_matrices(plan)) {
    const int64_t base = plan->tensors[mm.tensor].offset;
    const int64_t mat = mm.R * mm.C;
    if (mm.batch > 65535) return fail(VSF_ERR_ARG, "vsf_muon_step: more than 65535 matrices in a tensor");
    const dim3 grid(kMuonCtasPerMatrix, (unsigned)mm.batch);
    muon_momentum_kernel<<<grid, kMuonThreads, 0, st>>>(packed_grad, momentum, base, mat, mu,
                                                        partials);
    muon_scale_kernel<<<(unsigned)((mm.batch + 127) / 128), 128, 0, st>>>(
        partials, kMuonCtasPerMatrix, (int)mm.batch, hp->eps, r);
    muon_normalize_kernel<<<grid, kMuonThreads, 0, st>>>(packed_grad, momentum, base, mat, mu, r,
                                                         X);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return fail(VSF_ERR_CUDA, std::string("vsf_muon_step: ") + cudaGetErrorString(e));
    // Newton-Schulz, column-major view of the row-major R x C matrices: Xc is
    // C x R with leading dimension C.
    const bool tall = mm.R > mm.C;
    const int64_t n = std::min(mm.R, mm.C), sx = mat, sa = n * n;
    for (int it = 0; it < hp->ns_steps; ++it) {
      vsf_status s;
      // A (n x n) = X X^T (wide) or X^T X (tall)
      if (!tall)
        s = lt_gemm(true, false, n, n, mm.C, X, mm.C, sx, X, mm.C, sx, 1.0f, 0.0f, A, A, n, sa,
                    mm.batch, lt, st);
      else
        s = lt_gemm(false, true, n, n, mm.R, X, mm.C, sx, X, mm.C, sx, 1.0f, 0.0f, A, A, n, sa,
                    mm.batch, lt, st);
      if (s != VSF_OK) return s;
      // B = c A A + b A
      s = lt_gemm(false, false, n, n, n, A, n, sa, A, n, sa, nc, nb, A, B, n, sa, mm.batch, lt, st);
      if (s != VSF_OK) return s;
      // X' = a X + B X (wide) or a X + X B (tall), column-major Xc' = a Xc +
      // Xc B (wide) or a Xc + B Xc (tall)
      if (!tall)
        s = lt_gemm(false, false, mm.C, mm.R, mm.R, X, mm.C, sx, B, n, sa, 1.0f, na, X, Xn, mm.C,
                    sx, mm.batch, lt, st);
      else
        s = lt_gemm(false, false, mm.C, mm.R, mm.C, B, n, sa, X, mm.C, sx, 1.0f, na, X, Xn, mm.C,
                    sx, mm.batch, lt, st);
      if (s != VSF_OK) return s;
      std::swap(X, Xn);
    }
    const float alpha = (float)(hp->lr * std::sqrt(std::max(1.0, (double)mm.R / (double)mm.C)));
    const int64_t total = mm.batch * mat;
    const unsigned ugrid = (unsigned)std::min<int64_t>(4096, (total + kMuonThreads - 1) / kMuonThreads);
    muon_update_kernel<<<ugrid, kMuonThreads, 0, st>>>(X, master, packed_bf16, base, total, decay,
                                                       alpha);
    e = cudaGetLastError();
    if (e != cudaSuccess) return fail(VSF_ERR_CUDA, std::string("vsf_muon_step: ") + cudaGetErrorString(e));
  }
  return VSF_OK;
}

}  // extern "C"
