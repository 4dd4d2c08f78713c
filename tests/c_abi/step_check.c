/*
 * The shard step through the C ABI alone (include/vsf.h), with no Python and
 * no torch: plain cudaMalloc buffers, the four per-step calls for two steps,
 * and a byte-for-byte comparison with the oracle's C entry points on the
 * same inputs (layout, copy-in, factor, master, codes, scales, bf16 copy,
 * copy-out). Exit status 0 when everything matches.
 *
 * Three tensors on m = 4 virtual ranks, g_coll = 128: a 256 x 512 matrix in
 * 32-row blocks, a 300-element vector in element chunks and a 64 x 256
 * matrix in 32 x 32 tiles (the 2-D tensor-copy path).
 */
#include <math.h>
#include <stdint.h>
#include <stdio.h>
#include <stdlib.h>
#include <string.h>

#include <cuda_runtime_api.h>

#include "vsf.h"

/* The oracle's C entry points (test infrastructure, linked only here). */
int orc_plan(int n, const int64_t* rows, const int64_t* cols, const int32_t* gran,
             const int64_t* block_rows, const int64_t* tile_cols, int64_t m, int64_t g_coll,
             int policy, const int32_t* order, int64_t* S_out, int64_t* offsets_out);
int64_t orc_qblocks(int n, const int64_t* rows, const int64_t* cols, const int32_t* gran,
                    const int64_t* block_rows, const int64_t* tile_cols, int64_t g_coll,
                    const int64_t* offsets, int32_t* tensor_out, int64_t* base_out,
                    int64_t* nrows_out, int64_t* ncols_out, int64_t* stride_out);
void orc_pack(int n, const void* const* tensors, const int64_t* numel, const int64_t* offsets,
              int esize, void* packed);
void orc_unpack(int n, void* const* tensors, const int64_t* numel, const int64_t* offsets,
                int esize, const void* packed);
double orc_sumsq(int n, const void* const* tensors, const int64_t* numel, int is_bf16);
float orc_factor(double sumsq, int world, double max_norm, double* norm_out);
void orc_adam_all(int64_t nblocks, const int64_t* base, const int64_t* nrows, const int64_t* ncols,
                  const int64_t* stride, const void* packed_grad, int grad_bf16, float factor,
                  int quantized, void* m_state, void* v_state, float* m_scale, float* v_scale,
                  float* master, uint16_t* packed_bf16, double lr, double beta1, double beta2,
                  double eps, double wd, int step);

#define NT 3
#define M 4
#define GCOLL 128
#define STEPS 2

static int failures = 0;

static void check_status(vsf_status s, const char* what) {
  if (s != VSF_OK) {
    fprintf(stderr, "%s: %s (%s)\n", what, vsf_status_string(s), vsf_last_error());
    exit(2);
  }
}

static void check_cuda(cudaError_t e, const char* what) {
  if (e != cudaSuccess) {
    fprintf(stderr, "%s: %s\n", what, cudaGetErrorString(e));
    exit(2);
  }
}

static void same(const void* a, const void* b, size_t bytes, const char* what) {
  if (memcmp(a, b, bytes) != 0) {
    size_t i = 0;
    while (((const unsigned char*)a)[i] == ((const unsigned char*)b)[i]) ++i;
    fprintf(stderr, "MISMATCH %s at byte %zu of %zu\n", what, i, bytes);
    ++failures;
  }
}

/* fp32 -> bf16 bits, round to nearest even (inputs here are finite). */
static uint16_t to_bf16(float f) {
  uint32_t u;
  memcpy(&u, &f, 4);
  u += 0x7fffu + ((u >> 16) & 1u);
  return (uint16_t)(u >> 16);
}

int main(void) {
  const int64_t shape[NT][2] = {{256, 512}, {1, 300}, {64, 256}};
  const int32_t gran[NT] = {VSF_GRAN_ROWS, VSF_GRAN_ELEM, VSF_GRAN_TILE};
  const int64_t br[NT] = {32, 0, 32}, bc[NT] = {0, 0, 32};
  int64_t rows[NT], cols[NT], numel[NT];
  vsf_tensor_desc desc[NT];
  memset(desc, 0, sizeof(desc));
  for (int t = 0; t < NT; ++t) {
    rows[t] = shape[t][0];
    cols[t] = shape[t][1];
    numel[t] = rows[t] * cols[t];
    desc[t].ndim = t == 1 ? 1 : 2;
    if (t == 1) {
      desc[t].shape[0] = cols[t];
    } else {
      desc[t].shape[0] = rows[t];
      desc[t].shape[1] = cols[t];
    }
    desc[t].gran = gran[t];
    desc[t].block_rows = br[t];
    desc[t].tile_cols = bc[t];
  }

  /* ---- plan: library and oracle */
  vsf_plan* plan = NULL;
  check_status(vsf_plan_create(desc, NT, M, GCOLL, VSF_ORDER_DEFAULT, &plan), "vsf_plan_create");
  vsf_plan_info info;
  check_status(vsf_plan_get_info(plan, &info), "vsf_plan_get_info");
  int64_t off[NT], off_o[NT], S_o = 0;
  check_status(vsf_plan_offsets(plan, off), "vsf_plan_offsets");
  if (orc_plan(NT, rows, cols, gran, br, bc, M, GCOLL, 0, NULL, &S_o, off_o) != 0) {
    fprintf(stderr, "orc_plan failed\n");
    return 2;
  }
  if (S_o != info.S) ++failures, fprintf(stderr, "MISMATCH S %lld vs %lld\n", (long long)info.S, (long long)S_o);
  same(off, off_o, sizeof(off), "offsets");
  const int64_t total = info.total, nq = info.n_qblocks;
  int64_t nq_o = orc_qblocks(NT, rows, cols, gran, br, bc, GCOLL, off_o, NULL, NULL, NULL, NULL, NULL);
  if (nq_o != nq) {
    fprintf(stderr, "MISMATCH block count %lld vs %lld\n", (long long)nq, (long long)nq_o);
    return 1;
  }
  int32_t* qt = malloc(sizeof(int32_t) * nq);
  int64_t *qbase = malloc(8 * nq), *qr = malloc(8 * nq), *qc = malloc(8 * nq), *qs = malloc(8 * nq);
  orc_qblocks(NT, rows, cols, gran, br, bc, GCOLL, off_o, qt, qbase, qr, qc, qs);

  /* ---- inputs */
  uint16_t* grads[NT];
  float* masters[NT];
  for (int t = 0; t < NT; ++t) {
    grads[t] = malloc(2 * numel[t]);
    masters[t] = malloc(4 * numel[t]);
    for (int64_t i = 0; i < numel[t]; ++i) masters[t][i] = (float)(((i * 37 + t * 11) % 1001) - 500) * 1e-4f;
  }

  /* ---- device buffers (caller-owned) */
  size_t ws_bytes = vsf_plan_workspace_bytes(plan);
  void *d_ws, *d_grad, *d_bf, *d_m, *d_v;
  float *d_master, *d_msc, *d_vsc, *d_factor;
  double* d_norm;
  void* d_tgrad[NT];
  void* d_tparam[NT];
  check_cuda(cudaMalloc(&d_ws, ws_bytes), "cudaMalloc");
  check_cuda(cudaMalloc(&d_grad, 2 * total), "cudaMalloc");
  check_cuda(cudaMalloc((void**)&d_master, 4 * total), "cudaMalloc");
  check_cuda(cudaMalloc(&d_m, total), "cudaMalloc");
  check_cuda(cudaMalloc(&d_v, total), "cudaMalloc");
  check_cuda(cudaMalloc(&d_bf, 2 * total), "cudaMalloc");
  check_cuda(cudaMalloc((void**)&d_msc, 4 * nq), "cudaMalloc");
  check_cuda(cudaMalloc((void**)&d_vsc, 4 * nq), "cudaMalloc");
  check_cuda(cudaMalloc((void**)&d_factor, 16), "cudaMalloc");
  check_cuda(cudaMalloc((void**)&d_norm, 16), "cudaMalloc");
  for (int t = 0; t < NT; ++t) {
    check_cuda(cudaMalloc(&d_tgrad[t], 2 * numel[t]), "cudaMalloc");
    check_cuda(cudaMalloc(&d_tparam[t], 2 * numel[t]), "cudaMalloc");
  }
  void* zeros = calloc(4 * total, 1);
  check_cuda(cudaMemcpy(d_grad, zeros, 2 * total, cudaMemcpyHostToDevice), "zero");
  check_cuda(cudaMemcpy(d_master, zeros, 4 * total, cudaMemcpyHostToDevice), "zero");
  check_cuda(cudaMemcpy(d_m, zeros, total, cudaMemcpyHostToDevice), "zero");
  check_cuda(cudaMemcpy(d_v, zeros, total, cudaMemcpyHostToDevice), "zero");
  check_cuda(cudaMemcpy(d_bf, zeros, 2 * total, cudaMemcpyHostToDevice), "zero");
  check_cuda(cudaMemcpy(d_msc, zeros, 4 * nq, cudaMemcpyHostToDevice), "zero");
  check_cuda(cudaMemcpy(d_vsc, zeros, 4 * nq, cudaMemcpyHostToDevice), "zero");
  for (int t = 0; t < NT; ++t)
    check_cuda(cudaMemcpy(d_master + off[t], masters[t], 4 * numel[t], cudaMemcpyHostToDevice), "master");
  check_status(vsf_plan_upload(plan, d_ws, ws_bytes, NULL), "vsf_plan_upload");

  /* ---- oracle state */
  float* master_o = calloc(total, 4);
  int8_t* m_o = calloc(total, 1);
  uint8_t* v_o = calloc(total, 1);
  float *msc_o = calloc(nq, 4), *vsc_o = calloc(nq, 4);
  uint16_t* bf_o = calloc(total, 2);
  uint16_t* packed_o = calloc(total, 2);
  const void* mptrs[NT] = {masters[0], masters[1], masters[2]};
  orc_pack(NT, mptrs, numel, off_o, 4, master_o);

  vsf_adam_hparams hp = {1e-3, 0.9, 0.999, 1e-8, 0.01, INFINITY, M, 1};
  for (int step = 1; step <= STEPS; ++step) {
    for (int t = 0; t < NT; ++t) {
      for (int64_t i = 0; i < numel[t]; ++i)
        grads[t][i] = to_bf16((float)(((i * 7919 + t * 131 + step * 17) % 2001) - 1000) * 1e-6f);
      check_cuda(cudaMemcpy(d_tgrad[t], grads[t], 2 * numel[t], cudaMemcpyHostToDevice), "grad");
    }
    /* library: pack, group norm / scale, 8-bit AdamW, unpack */
    check_status(vsf_pack(plan, (const void* const*)d_tgrad, VSF_BF16, d_grad, NULL), "vsf_pack");
    check_status(vsf_group_norm_scale(plan, NULL, VSF_BF16, &hp, d_factor, d_norm, NULL),
                 "vsf_group_norm_scale");
    check_status(vsf_adam8_step(plan, d_grad, VSF_BF16, d_factor, d_master, d_m, d_v, d_msc, d_vsc,
                                (uint16_t*)d_bf, &hp, step, NULL), "vsf_adam8_step");
    check_status(vsf_unpack(plan, (const uint16_t*)d_bf, d_tparam, NULL), "vsf_unpack");
    check_cuda(cudaDeviceSynchronize(), "step");

    /* oracle: the same step */
    const void* gptrs[NT] = {grads[0], grads[1], grads[2]};
    orc_pack(NT, gptrs, numel, off_o, 2, packed_o);
    double norm_o = 0.0;
    const float factor_o = orc_factor(orc_sumsq(NT, gptrs, numel, 1), M, INFINITY, &norm_o);
    orc_adam_all(nq, qbase, qr, qc, qs, packed_o, 1, factor_o, 1, m_o, v_o, msc_o, vsc_o, master_o,
                 bf_o, hp.lr, hp.beta1, hp.beta2, hp.eps, hp.weight_decay, step);

    float factor = 0.0f;
    check_cuda(cudaMemcpy(&factor, d_factor, 4, cudaMemcpyDeviceToHost), "factor");
    same(&factor, &factor_o, 4, "factor");
  }

  /* ---- compare every buffer */
  void* host = malloc(4 * total);
  check_cuda(cudaMemcpy(host, d_grad, 2 * total, cudaMemcpyDeviceToHost), "copy");
  same(host, packed_o, 2 * total, "packed gradient (copy-in)");
  check_cuda(cudaMemcpy(host, d_master, 4 * total, cudaMemcpyDeviceToHost), "copy");
  same(host, master_o, 4 * total, "master");
  check_cuda(cudaMemcpy(host, d_m, total, cudaMemcpyDeviceToHost), "copy");
  same(host, m_o, total, "m codes");
  check_cuda(cudaMemcpy(host, d_v, total, cudaMemcpyDeviceToHost), "copy");
  same(host, v_o, total, "v codes");
  check_cuda(cudaMemcpy(host, d_msc, 4 * nq, cudaMemcpyDeviceToHost), "copy");
  same(host, msc_o, 4 * nq, "m scales");
  check_cuda(cudaMemcpy(host, d_vsc, 4 * nq, cudaMemcpyDeviceToHost), "copy");
  same(host, vsc_o, 4 * nq, "v scales");
  check_cuda(cudaMemcpy(host, d_bf, 2 * total, cudaMemcpyDeviceToHost), "copy");
  same(host, bf_o, 2 * total, "bf16 parameters");
  uint16_t* params_o[NT];
  for (int t = 0; t < NT; ++t) params_o[t] = malloc(2 * numel[t]);
  orc_unpack(NT, (void* const*)params_o, numel, off_o, 2, bf_o);
  for (int t = 0; t < NT; ++t) {
    check_cuda(cudaMemcpy(host, d_tparam[t], 2 * numel[t], cudaMemcpyDeviceToHost), "copy");
    same(host, params_o[t], 2 * numel[t], "copy-out");
  }

  vsf_plan_destroy(plan);
  printf("%s: S=%lld, %lld quantisation blocks, %d steps\n", failures ? "MISMATCH" : "bit-exact",
         (long long)info.S, (long long)nq, STEPS);
  return failures ? 1 : 0;
}
