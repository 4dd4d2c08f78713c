// ns_gemm.cuh — the Newton–Schulz products of distributed Muon on the
// fifth-generation tensor cores (tcgen05, sm_103a). Included by muon.cu
// inside namespace vsf::{anonymous}, after mbarrier.cuh.
//
// Method: "veScale-FSDP: Flexible and High-Performance FSDP at Scale (MLSys
// 2026)" summary page › 结构感知训练 case study › 分布式 Muon (Algorithm 2):
// the root rank orthogonalises a whole matrix by Newton–Schulz, three
// products per iteration: the Gram matrix A = X X^T (or X^T X), B = c A A +
// b A, and X' = a X + B X (or a X + X B).
//
// One launch computes, for every matrix b of a strided batch,
//   D[b] = alpha * opA[b] * opB[b]^T + beta * C[b]
// with opA M x K and opB N x K, bf16 operands and output, fp32 accumulation
// in tensor memory (TMEM). Each operand is stored either K-major (row i at
// ptr + i*ld, K contiguous) or MN-major (row k at ptr + k*ld, M or N
// contiguous), so that X^T X and B X need no transposed copy.
//
// Symmetric products (SYM: opA = opB, so D = D^T up to beta * C with C
// symmetric) compute only the output tiles that reach the diagonal or lie
// above it, half of the FLOPs. The epilogue writes every element (i, j) with
// i <= j to D[i][j] and D[j][i]; elements below the diagonal are never
// written directly, so D comes out exactly symmetric.
//
// CTA structure (persistent: one CTA per SM, tiles round-robin):
//   warp 0      TMA producer: 64-element K slices of both operands into a
//               4-stage ring of 48 KB stages (128-byte swizzle), each stage
//               guarded by a "full" mbarrier (transaction bytes) and an
//               "empty" mbarrier (arrived by the MMAs' commit);
//   warp 1      allocates 512 TMEM columns (two 128 x 256 fp32
//               accumulators); one thread issues tcgen05.mma (M = 128,
//               N = 256, K = 16 per instruction) and commits each stage back
//               to the producer and each finished accumulator to the
//               epilogue;
//   warps 2..5  epilogue: tcgen05.ld of their 32-lane quarter of the
//               accumulator, alpha * acc + beta * C in fp32, bf16 round to
//               nearest even, stores (and mirrored stores). The two
//               accumulators let the epilogue of one tile overlap the MMAs
//               of the next.
// Clusters of two (CL = 2): the two CTAs of a cluster compute vertically
// adjacent tiles (rows m0 and m0 + 128, the same 256 columns), so they need
// the same opB slice every stage. Each loads its own opA slice and half of
// the opB slice, multicast into both CTAs' shared memory: 32 KB of L2 reads
// per CTA and stage instead of 48. A stage is refilled only when both CTAs'
// MMAs are done with it (each MMA commit arrives on both CTAs' "empty"
// barriers).
//
// Every wait is bounded (mbarrier.cuh): a broken pipeline sets bit 1 of the
// device error word and the kernel ends (a timeout also stops the cluster
// peer); before exit the producer waits for its issued copies and the MMA
// thread for its issued MMAs, the cluster synchronises, and TMEM is freed.

constexpr int kGemmBM = 128;   // rows of an output tile (TMEM lanes)
constexpr int kGemmBN = 256;   // columns of an output tile (TMEM columns)
constexpr int kGemmBK = 64;    // K elements per stage: one 128-byte swizzle row
constexpr int kGemmStages = 4;
constexpr uint32_t kGemmABytes = kGemmBM * kGemmBK * 2;  // 16 KB
constexpr uint32_t kGemmBBytes = kGemmBN * kGemmBK * 2;  // 32 KB
constexpr uint32_t kGemmStageBytes = kGemmABytes + kGemmBBytes;
constexpr int kGemmThreads = 192;
constexpr uint32_t kGemmBarBytes = 8 * (2 * kGemmStages + 5);
// +1024: the kernel rounds the dynamic shared memory base up to 1024 bytes
// (the 128-byte swizzle repeats every 1024 bytes)
constexpr uint32_t kGemmSmem = kGemmStages * kGemmStageBytes + kGemmBarBytes + 1024;
static_assert(kGemmSmem <= 227 * 1024, "GEMM ring fits in shared memory");

struct NsGemmArgs {
  int M, N, K, batch;
  float alpha, beta;
  const uint16_t* C;  // read when beta != 0
  int64_t ldc, sc;
  uint16_t* D;
  int64_t ldd, sd;
  int tiles_per_matrix;  // work items per matrix: tiles (CL = 1) or vertical tile pairs (CL = 2)
  int mgroups;           // row groups per matrix: 128-row blocks (CL = 1) or 256-row pairs
};

// ---------------------------------------------------------------- PTX wrappers

__device__ __forceinline__ void tmem_alloc(uint32_t dst_smem, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(dst_smem),
               "r"(ncols)
               : "memory");
}
__device__ __forceinline__ void tmem_relinquish() {
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
               : "memory");
}
__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// D (TMEM) (+)= A (shared) * B (shared)^T, kind::f16 (bf16 here), one thread.
__device__ __forceinline__ void umma_bf16(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc,
                                          uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
      " tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// The mbarrier receives one arrival once every tcgen05 operation this thread
// issued before has completed.
__device__ __forceinline__ void umma_commit(uint32_t bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
                   bar)
               : "memory");
}

// 32 consecutive fp32 columns of this thread's TMEM lane.
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, "
      "%12, %13, %14, %15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, "
      "%30, %31}, [%32];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
        "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]),
        "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]),
        "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr));
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}

// 3-D tensor copy (global -> shared) of one box at (x, y, z), completing on bar.
__device__ __forceinline__ void tma3_g2s(uint32_t dst, const CUtensorMap* map, int x, int y, int z,
                                         uint32_t bar) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3, %4}], [%5];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(z), "r"(bar)
      : "memory");
}

// The same box written to the same shared-memory offset of every CTA in
// cta_mask (cluster ranks), each CTA's mbarrier at `bar` receiving its bytes.
__device__ __forceinline__ void tma3_g2s_multicast(uint32_t dst, const CUtensorMap* map, int x, int y,
                                                   int z, uint32_t bar, uint16_t cta_mask) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.mbarrier::complete_tx::bytes"
      ".multicast::cluster [%0], [%1, {%2, %3, %4}], [%5], %6;" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(z), "r"(bar), "h"(cta_mask)
      : "memory");
}

// tcgen05.commit arriving on the mbarrier at `bar` in every CTA of cta_mask.
__device__ __forceinline__ void umma_commit_multicast(uint32_t bar, uint16_t cta_mask) {
  asm volatile(
      "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64"
      " [%0], %1;" ::"r"(bar),
      "h"(cta_mask)
      : "memory");
}

// Sets the stop flag at the same shared-memory offset in cluster rank `rank`.
__device__ __forceinline__ void remote_stop(volatile uint32_t* stop, uint32_t rank) {
  uint32_t ra;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;"
               : "=r"(ra)
               : "r"(smem_u32(const_cast<uint32_t*>(stop))), "r"(rank));
  asm volatile("st.shared::cluster.u32 [%0], %1;" ::"r"(ra), "r"(1u) : "memory");
}

__device__ __forceinline__ uint32_t cluster_rank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}
__device__ __forceinline__ void cluster_barrier() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::
                   : "memory");
}

// Shared-memory matrix descriptor of tcgen05 (128-byte swizzle): start
// address, leading- and stride-dimension byte offsets (all >> 4), the fixed
// version bits 46-48 = 0b001, swizzle mode 2 (128B) in bits 61-63.
__host__ __device__ constexpr uint64_t umma_smem_desc(uint32_t addr, uint32_t lbo, uint32_t sbo) {
  return (uint64_t)((addr & 0x3FFFFu) >> 4) | ((uint64_t)((lbo >> 4) & 0x3FFFu) << 16) |
         ((uint64_t)((sbo >> 4) & 0x3FFFu) << 32) | (1ull << 46) | (2ull << 61);
}

// Instruction descriptor of kind::f16: fp32 accumulator (bits 4-5 = 1), bf16
// A and B (bits 7-9, 10-12 = 1), A / B MN-major flags (bits 15, 16), N >> 3
// (bits 17-22), M >> 4 (bits 24-28).
__host__ __device__ constexpr uint32_t umma_idesc_bf16(bool a_mn, bool b_mn, int m, int n) {
  return (1u << 4) | (1u << 7) | (1u << 10) | ((a_mn ? 1u : 0u) << 15) |
         ((b_mn ? 1u : 0u) << 16) | ((uint32_t)(n >> 3) << 17) | ((uint32_t)(m >> 4) << 24);
}

// Operand layouts in a stage (both from 128-byte-swizzled tensor copies):
//   K-major, R rows x 64 K: row r at r * 128 bytes; 8-row groups 1024 bytes
//     apart (stride offset); one MMA's 16 K elements are 32 bytes of each
//     row, so K step kk starts kk * 32 bytes in.
//   MN-major, 64 K rows x R: boxes of 64 MN elements x 64 K rows, 8 KB each,
//     side by side (leading offset 8192 between 64-element MN groups); K row
//     k at k * 128 bytes in its box, 8-row groups 1024 bytes apart; K step kk
//     starts kk * 16 rows = kk * 2048 bytes in.
template <bool kMN>
__device__ __forceinline__ uint64_t operand_desc(uint32_t base, int kk) {
  return kMN ? umma_smem_desc(base + kk * 2048u, 8192u, 1024u)
             : umma_smem_desc(base + kk * 32u, 16u, 1024u);
}

__device__ __forceinline__ int imin(int a, int b) { return a < b ? a : b; }

// Work item t of the launch: matrix b, first row m0 of this CTA's tile
// (rank: its position in a cluster of CL vertically adjacent tiles), first
// column n0. Items run column block by column block (consecutive items share
// the opB panel); a symmetric product keeps, in column block J (columns
// 256J .. 256J+255), the row blocks 0 .. 2J+1 that reach the diagonal, i.e.
// the 128-row groups 0 .. 2J+1 (CL = 1) or the 256-row groups 0 .. J (CL = 2).
template <int CL>
__device__ __forceinline__ void gemm_tile(const NsGemmArgs& g, bool sym, int t, int rank, int& b,
                                          int& m0, int& n0) {
  b = t / g.tiles_per_matrix;
  int r = t - b * g.tiles_per_matrix;
  if (!sym) {
    const int J = r / g.mgroups;
    m0 = (r - J * g.mgroups) * (kGemmBM * CL) + rank * kGemmBM;
    n0 = J * kGemmBN;
    return;
  }
  int J = 0;
  for (;;) {
    const int cnt = imin(g.mgroups, CL == 1 ? 2 * J + 2 : J + 1);
    if (r < cnt) break;
    r -= cnt;
    ++J;
  }
  m0 = r * (kGemmBM * CL) + rank * kGemmBM;
  n0 = J * kGemmBN;
}

__device__ __forceinline__ uint16_t bf16_rn(float x) {
  const __nv_bfloat16 h = __float2bfloat16_rn(x);
  return *reinterpret_cast<const uint16_t*>(&h);
}

template <bool AMN, bool BMN, bool SYM, int CL>
__global__ void __launch_bounds__(kGemmThreads, 1)
    ns_gemm_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                   const NsGemmArgs g, unsigned* err) {
  static_assert(CL == 1 || CL == 2, "clusters of one or two CTAs");
  extern __shared__ __align__(1024) unsigned char gsm_raw[];
  unsigned char* sm = gsm_raw + ((1024u - (smem_u32(gsm_raw) & 1023u)) & 1023u);
  const uint32_t s0 = smem_u32(sm);
  const uint32_t bar0 = s0 + kGemmStages * kGemmStageBytes;
  auto full_bar = [&](int s) { return bar0 + 8u * s; };
  auto empty_bar = [&](int s) { return bar0 + 8u * (kGemmStages + s); };
  auto tfull_bar = [&](int i) { return bar0 + 8u * (2 * kGemmStages + i); };
  auto tempty_bar = [&](int i) { return bar0 + 8u * (2 * kGemmStages + 2 + i); };
  const uint32_t done_bar = bar0 + 8u * (2 * kGemmStages + 4);
  __shared__ uint32_t tmem_slot;
  __shared__ uint32_t stop_flag;
  volatile uint32_t* stop = &stop_flag;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int rank = CL == 1 ? 0 : (int)cluster_rank();
  const int cid = blockIdx.x / CL, ncid = gridDim.x / CL;
  constexpr uint16_t kBoth = (1u << CL) - 1u;  // every CTA of the cluster

  if (threadIdx.x == 0) {
    stop_flag = 0u;
    for (int s = 0; s < kGemmStages; ++s) {
      mbar_init(full_bar(s), 1);
      mbar_init(empty_bar(s), CL);  // one MMA commit from each CTA of the cluster
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(tfull_bar(i), 1);
      mbar_init(tempty_bar(i), 4);  // one arrival per epilogue warp
    }
    mbar_init(done_bar, 1);
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(&tmem_slot), 512);
    tmem_relinquish();
  }
  tc_fence_before();
  if (CL > 1)
    cluster_barrier();  // the peer's barriers exist before any multicast signals them
  else
    __syncthreads();
  tc_fence_after();
  const uint32_t tmem = tmem_slot;
  const int ntiles = g.batch * g.tiles_per_matrix;
  const int KB = (g.K + kGemmBK - 1) / kGemmBK;
  // a timeout here also stops the cluster peer, which would otherwise keep
  // multicasting into this CTA
  auto halt_cluster = [&]() {
    if (CL > 1) remote_stop(stop, (uint32_t)(rank ^ 1));
  };

  if (warp == 0) {
    if (lane == 0) {
      // ---------------- producer
      uint32_t it = 0;  // stages issued
      bool halted = false;
      for (int t = cid; t < ntiles && !halted; t += ncid) {
        int b, m0, n0;
        gemm_tile<CL>(g, SYM, t, rank, b, m0, n0);
        for (int kb = 0; kb < KB; ++kb) {
          const int s = it % kGemmStages;
          const uint32_t ph = (it / kGemmStages) & 1u;
          if (!mbar_wait(empty_bar(s), ph ^ 1u, err, stop)) {
            halted = true;
            halt_cluster();
            break;
          }
          ++it;
          mbar_expect_tx(full_bar(s), kGemmStageBytes);
          const uint32_t a = s0 + s * kGemmStageBytes, bb = a + kGemmABytes;
          const int k0 = kb * kGemmBK;
          if (AMN) {
            tma3_g2s(a, &tmA, m0, k0, b, full_bar(s));
            tma3_g2s(a + 8192u, &tmA, m0 + 64, k0, b, full_bar(s));
          } else {
            tma3_g2s(a, &tmA, k0, m0, b, full_bar(s));
          }
          if (CL == 1) {
            if (BMN) {
              for (int h = 0; h < 4; ++h)
                tma3_g2s(bb + h * 8192u, &tmB, n0 + 64 * h, k0, b, full_bar(s));
            } else {
              tma3_g2s(bb, &tmB, k0, n0, b, full_bar(s));
            }
          } else {
            // this CTA's half of the opB slice, into both CTAs
            if (BMN) {
              for (int h = 2 * rank; h < 2 * rank + 2; ++h)
                tma3_g2s_multicast(bb + h * 8192u, &tmB, n0 + 64 * h, k0, b, full_bar(s), kBoth);
            } else {
              tma3_g2s_multicast(bb + rank * (kGemmBBytes / 2), &tmB, k0, n0 + rank * (kGemmBN / 2),
                                 b, full_bar(s), kBoth);
            }
          }
        }
      }
      // every issued copy lands before the CTA exits (one limit in all)
      const uint64_t deadline = global_ns() + kWaitNs;
      for (int s = 0; s < kGemmStages; ++s) {
        if (it > (uint32_t)s) {
          const uint32_t last = (it - 1 - s) / kGemmStages * kGemmStages + s;
          mbar_drain(full_bar(s), (last / kGemmStages) & 1u, deadline, err);
        }
      }
    }
  } else if (warp == 1) {
    if (lane == 0) {
      // ---------------- MMA issuer
      constexpr uint32_t idesc = umma_idesc_bf16(AMN, BMN, kGemmBM, kGemmBN);
      uint32_t it = 0;
      int lt = 0;
      bool halted = false;
      for (int t = cid; t < ntiles && !halted; t += ncid, ++lt) {
        const int buf = lt & 1;
        if (!mbar_wait(tempty_bar(buf), ((uint32_t)(lt >> 1) & 1u) ^ 1u, err, stop)) {
          halt_cluster();
          break;
        }
        tc_fence_after();
        const uint32_t d = tmem + (uint32_t)(buf * kGemmBN);
        for (int kb = 0; kb < KB; ++kb, ++it) {
          const int s = it % kGemmStages;
          if (!mbar_wait(full_bar(s), (it / kGemmStages) & 1u, err, stop)) {
            halted = true;
            halt_cluster();
            break;
          }
          tc_fence_after();
          const uint32_t a = s0 + s * kGemmStageBytes, bb = a + kGemmABytes;
#pragma unroll
          for (int kk = 0; kk < kGemmBK / 16; ++kk)
            umma_bf16(d, operand_desc<AMN>(a, kk), operand_desc<BMN>(bb, kk), idesc,
                      (kb | kk) != 0 ? 1u : 0u);
          // the stage is free once these MMAs are done, in this CTA and (its
          // opB half lives in both) in the peer
          if (CL == 1)
            umma_commit(empty_bar(s));
          else
            umma_commit_multicast(empty_bar(s), kBoth);
        }
        if (!halted) umma_commit(tfull_bar(buf));  // the accumulator is complete
      }
      // every issued MMA completes before TMEM is freed
      umma_commit(done_bar);
      mbar_drain(done_bar, 0u, global_ns() + kWaitNs, err);
    }
  } else {
    // ---------------- epilogue: warp w reads TMEM lanes 32 (w % 4) .. + 31
    const int q = warp & 3;
    int lt = 0;
    for (int t = cid; t < ntiles; t += ncid, ++lt) {
      const int buf = lt & 1;
      const bool ok =
          __all_sync(0xffffffffu, mbar_wait(tfull_bar(buf), (uint32_t)(lt >> 1) & 1u, err, stop));
      tc_fence_after();
      if (ok) {
        int b, m0, n0;
        gemm_tile<CL>(g, SYM, t, rank, b, m0, n0);
        const int i = m0 + 32 * q + lane;  // this thread's output row
        const bool row_ok = i < g.M;
        uint16_t* Db = g.D + (int64_t)b * g.sd;
        const uint16_t* Cb = g.beta != 0.0f ? g.C + (int64_t)b * g.sc : nullptr;
#pragma unroll 1
        for (int c = 0; c < kGemmBN / 32; ++c) {
          const int j0 = n0 + 32 * c;
          uint32_t r[32];
          __syncwarp();  // tcgen05.ld is warp-collective: reconverge after a lane's `continue`
          tmem_ld32(tmem + (uint32_t)(buf * kGemmBN + 32 * c) + ((uint32_t)(32 * q) << 16), r);
          if (!row_ok || j0 >= g.N) continue;
          if (SYM && j0 + 31 < i) continue;  // the whole chunk lies below the diagonal
          const bool full = j0 + 32 <= g.N;
          float v[32];
#pragma unroll
          for (int x = 0; x < 32; ++x) v[x] = __fmul_rn(g.alpha, __uint_as_float(r[x]));
          if (Cb != nullptr) {
            const uint16_t* crow = Cb + (int64_t)i * g.ldc + j0;
            if (full) {
#pragma unroll
              for (int w = 0; w < 4; ++w) {
                const uint4 u = *reinterpret_cast<const uint4*>(crow + 8 * w);
                const uint32_t wd[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
                for (int h = 0; h < 4; ++h) {
                  v[8 * w + 2 * h] = __fmaf_rn(g.beta, __uint_as_float(wd[h] << 16), v[8 * w + 2 * h]);
                  v[8 * w + 2 * h + 1] =
                      __fmaf_rn(g.beta, __uint_as_float(wd[h] & 0xffff0000u), v[8 * w + 2 * h + 1]);
                }
              }
            } else {
#pragma unroll
              for (int x = 0; x < 32; ++x)
                if (j0 + x < g.N)
                  v[x] = __fmaf_rn(g.beta, __uint_as_float((uint32_t)crow[x] << 16), v[x]);
            }
          }
          uint16_t* drow = Db + (int64_t)i * g.ldd + j0;
          if (full && (!SYM || j0 >= i)) {
#pragma unroll
            for (int w = 0; w < 4; ++w) {
              uint32_t wd[4];
#pragma unroll
              for (int h = 0; h < 4; ++h)
                wd[h] = (uint32_t)bf16_rn(v[8 * w + 2 * h]) |
                        ((uint32_t)bf16_rn(v[8 * w + 2 * h + 1]) << 16);
              *reinterpret_cast<uint4*>(drow + 8 * w) = make_uint4(wd[0], wd[1], wd[2], wd[3]);
            }
          } else {
#pragma unroll
            for (int x = 0; x < 32; ++x)
              if (j0 + x < g.N && (!SYM || j0 + x >= i)) drow[x] = bf16_rn(v[x]);
          }
          if (SYM) {
            // mirror: D[j][i] for j > i (lanes write consecutive i: coalesced)
#pragma unroll
            for (int x = 0; x < 32; ++x) {
              const int j = j0 + x;
              if (j > i && j < g.N) Db[(int64_t)j * g.ldd + i] = bf16_rn(v[x]);
            }
          }
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(tempty_bar(buf));
    }
  }
  tc_fence_before();
  __syncthreads();
  // neither CTA of a cluster leaves while its peer may still write into it
  if (CL > 1) cluster_barrier();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

// Plain CUDA-core GEMM of the same contract for operands the tensor copies
// cannot address (a leading dimension or batch stride that is not a
// multiple of 8 elements, or an address not on 16 bytes): one thread per
// output element, fp32 accumulation in K order. Only small matrices take it.
template <bool AMN, bool BMN, bool SYM>
__global__ void __launch_bounds__(256) ns_gemm_simt_kernel(const uint16_t* __restrict__ A,
                                                           int64_t lda, int64_t sa,
                                                           const uint16_t* __restrict__ B,
                                                           int64_t ldb, int64_t sb,
                                                           const NsGemmArgs g) {
  const int j = blockIdx.x * 16 + (threadIdx.x & 15);
  const int i = blockIdx.y * 16 + (threadIdx.x >> 4);
  const int b = blockIdx.z;
  if (i >= g.M || j >= g.N || (SYM && i > j)) return;
  const uint16_t* Ab = A + (int64_t)b * sa;
  const uint16_t* Bb = B + (int64_t)b * sb;
  float acc = 0.0f;
  for (int k = 0; k < g.K; ++k) {
    const float x = __uint_as_float((uint32_t)(AMN ? Ab[(int64_t)k * lda + i] : Ab[(int64_t)i * lda + k]) << 16);
    const float y = __uint_as_float((uint32_t)(BMN ? Bb[(int64_t)k * ldb + j] : Bb[(int64_t)j * ldb + k]) << 16);
    acc = __fmaf_rn(x, y, acc);
  }
  float v = __fmul_rn(g.alpha, acc);
  if (g.beta != 0.0f)
    v = __fmaf_rn(g.beta, __uint_as_float((uint32_t)g.C[(int64_t)b * g.sc + (int64_t)i * g.ldc + j] << 16), v);
  uint16_t* Db = g.D + (int64_t)b * g.sd;
  Db[(int64_t)i * g.ldd + j] = bf16_rn(v);
  if (SYM && i != j) Db[(int64_t)j * g.ldd + i] = bf16_rn(v);
}
