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
// Pair MMA: the two CTAs of a cluster compute one 256 x 256 output tile with
// tcgen05.mma.cta_group::2 (M = 256 across the pair, N = 256, K = 16). Each
// CTA stages only its own 128 rows of opA and its own 128 rows of opB per
// 64-element K slice (32 KB), so each SM's shared memory serves half of the
// opB reads and a 6-stage ring fits. (A single-SM 128 x 256 tile needs 48 KB
// per slice, written by the copies and read by the tensor core, about 190
// bytes per clock through one SM's shared memory at the tensor rate; measured,
// it kept the tensor pipe 74-79% busy and ran 8-20% slower.) Each CTA's
// accumulator, its 128 rows x 256 columns, lives in its own TMEM.
//
// CTA structure (persistent: one cluster per SM pair, tiles round-robin):
//   warp 0      TMA producer, in both CTAs: this CTA's opA and opB rows of
//               each K slice (128-byte swizzle); the copies of both CTAs
//               signal the leader's "full" barrier (.cta_group::2 copies),
//               on which the leader posts the pair's byte count;
//   warp 1      allocates 512 TMEM columns (two accumulators) in both CTAs;
//               one thread of the leader (cluster rank 0) issues every MMA
//               and commits each stage to both CTAs' "empty" barriers and
//               each finished accumulator to both CTAs' "accumulator full"
//               barriers (multicast);
//   warps 2..5  epilogue, in both CTAs: tcgen05.ld of their 32-lane quarter
//               of this CTA's accumulator, alpha * acc + beta * C in fp32,
//               bf16 round to nearest even, stores (and mirrored stores);
//               then an arrival on the leader's "accumulator empty" barrier.
//               The two accumulators let the epilogue of one tile overlap
//               the MMAs of the next.
// Every wait is bounded (mbarrier.cuh): a broken pipeline sets bit 1 of the
// device error word and stops both CTAs of the pair; the leader waits for
// the pair's copies and its MMAs before exit, and the pair synchronises
// before TMEM is freed. A pair whose two TMEM allocations differ in address
// (the leader's MMAs write both at the leader's) sets bit 3 and computes
// nothing.

constexpr int kGemmBM = 128;   // rows of a CTA's half of the output tile (TMEM lanes)
constexpr int kGemmBN = 256;   // columns of an output tile (TMEM columns)
constexpr int kGemmBK = 64;    // K elements per stage: one 128-byte swizzle row
constexpr int kGemmStages = 6;
constexpr uint32_t kGemmABytes = kGemmBM * kGemmBK * 2;        // 16 KB: this CTA's opA rows
constexpr uint32_t kGemmBBytes = (kGemmBN / 2) * kGemmBK * 2;  // 16 KB: this CTA's opB rows
constexpr uint32_t kGemmStageBytes = kGemmABytes + kGemmBBytes;
constexpr uint32_t kGemmTmemCols = 2 * kGemmBN;               // two fp32 accumulators
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
  int tiles_per_matrix;  // 256 x 256 output tiles per matrix
  int mgroups;           // 256-row groups per matrix
};

// ---------------------------------------------------------------- PTX wrappers

// TMEM allocation of the CTA pair: one warp of each CTA executes it, and the
// pair gets `ncols` columns at the same address in both CTAs' TMEM.
__device__ __forceinline__ void tmem_alloc_pair(uint32_t dst_smem, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(dst_smem),
               "r"(ncols)
               : "memory");
}
__device__ __forceinline__ void tmem_relinquish_pair() {
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc_pair(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
               : "memory");
}
__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// D (both CTAs' TMEM) (+)= A (both CTAs' shared memory) * B^T, kind::f16
// (bf16 here), issued by one thread of the leader CTA.
__device__ __forceinline__ void umma_pair_bf16(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc,
                                               uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
      " tcgen05.mma.cta_group::2.kind::f16 [%0], %1, %2, %3, p;\n}" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// The mbarrier at `bar` in every CTA of cta_mask receives one arrival once
// every pair MMA this thread issued before has completed.
__device__ __forceinline__ void umma_pair_commit(uint32_t bar, uint16_t cta_mask) {
  asm volatile(
      "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64"
      " [%0], %1;" ::"r"(bar),
      "h"(cta_mask)
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

// 3-D tensor copy (global -> this CTA's shared memory) of one box at
// (x, y, z), completing on an mbarrier of either CTA of the pair (bar: a
// shared::cluster address).
__device__ __forceinline__ void tma3_g2s_pair(uint32_t dst, const CUtensorMap* map, int x, int y,
                                              int z, uint32_t bar) {
  asm volatile(
      "cp.async.bulk.tensor.3d.cta_group::2.shared::cluster.global.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3, %4}], [%5];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(z), "r"(bar)
      : "memory");
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
// The shared::cluster address of the same offset in cluster rank `rank`.
__device__ __forceinline__ uint32_t peer_addr(uint32_t local, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(local), "r"(rank));
  return r;
}
__device__ __forceinline__ uint32_t ld_peer_u32(uint32_t cluster_addr) {
  uint32_t v;
  asm volatile("ld.shared::cluster.u32 %0, [%1];" : "=r"(v) : "r"(cluster_addr) : "memory");
  return v;
}
// Sets the stop flag at the same shared-memory offset in cluster rank `rank`.
__device__ __forceinline__ void remote_stop(volatile uint32_t* stop, uint32_t rank) {
  asm volatile("st.shared::cluster.u32 [%0], %1;" ::"r"(
                   peer_addr(smem_u32(const_cast<uint32_t*>(stop)), rank)),
               "r"(1u)
               : "memory");
}
// Arrival on an mbarrier of the cluster (release at cluster scope).
__device__ __forceinline__ void mbar_arrive_cluster(uint32_t cluster_addr) {
  asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(cluster_addr)
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

// Operand layouts in a stage (both from 128-byte-swizzled tensor copies of
// this CTA's 128 rows):
//   K-major, 128 rows x 64 K: row r at r * 128 bytes; 8-row groups 1024 bytes
//     apart (stride offset); one MMA's 16 K elements are 32 bytes of each
//     row, so K step kk starts kk * 32 bytes in.
//   MN-major, 64 K rows x 128: two boxes of 64 MN elements x 64 K rows, 8 KB
//     each, side by side (leading offset 8192 between 64-element MN groups);
//     K row k at k * 128 bytes in its box, 8-row groups 1024 bytes apart; K
//     step kk starts kk * 16 rows = kk * 2048 bytes in.
template <bool kMN>
__device__ __forceinline__ uint64_t operand_desc(uint32_t base, int kk) {
  return kMN ? umma_smem_desc(base + kk * 2048u, 8192u, 1024u)
             : umma_smem_desc(base + kk * 32u, 16u, 1024u);
}

__device__ __forceinline__ int imin(int a, int b) { return a < b ? a : b; }

// Work item t of the launch: matrix b, and the 256 x 256 output tile whose
// 128-row half this CTA (cluster rank `rank`) holds: first row m0, first
// column n0. Items run column block by column block (consecutive items share
// the opB panel); a symmetric product keeps, in column block J (columns
// 256J .. 256J+255), the 256-row groups 0 .. J that reach the diagonal.
__device__ __forceinline__ void gemm_tile(const NsGemmArgs& g, bool sym, int t, int rank, int& b,
                                          int& m0, int& n0) {
  b = t / g.tiles_per_matrix;
  int r = t - b * g.tiles_per_matrix;
  if (!sym) {
    const int J = r / g.mgroups;
    m0 = (r - J * g.mgroups) * (2 * kGemmBM) + rank * kGemmBM;
    n0 = J * kGemmBN;
    return;
  }
  int J = 0;
  for (;;) {
    const int cnt = imin(g.mgroups, J + 1);
    if (r < cnt) break;
    r -= cnt;
    ++J;
  }
  m0 = r * (2 * kGemmBM) + rank * kGemmBM;
  n0 = J * kGemmBN;
}

__device__ __forceinline__ uint16_t bf16_rn(float x) {
  const __nv_bfloat16 h = __float2bfloat16_rn(x);
  return *reinterpret_cast<const uint16_t*>(&h);
}

template <bool AMN, bool BMN, bool SYM>
__global__ void __launch_bounds__(kGemmThreads, 1)
    ns_gemm_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                   const NsGemmArgs g, unsigned* err) {
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
  const int rank = (int)cluster_rank();
  const bool leader = rank == 0;
  const int cid = blockIdx.x / 2, ncid = gridDim.x / 2;
  constexpr uint16_t kBoth = 3;

  if (threadIdx.x == 0) {
    stop_flag = 0u;
    for (int s = 0; s < kGemmStages; ++s) {
      mbar_init(full_bar(s), 1);   // the leader's producer posts both CTAs' bytes
      mbar_init(empty_bar(s), 1);  // the leader's MMA commit
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(tfull_bar(i), 1);
      mbar_init(tempty_bar(i), 8);  // every epilogue warp of both CTAs (leader's barrier)
    }
    mbar_init(done_bar, 1);
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  if (warp == 1) {
    tmem_alloc_pair(smem_u32(&tmem_slot), kGemmTmemCols);
    tmem_relinquish_pair();
  }
  tc_fence_before();
  cluster_barrier();
  tc_fence_after();
  const uint32_t tmem = tmem_slot;
  // the leader's MMAs write both CTAs' accumulators at the leader's address
  if (threadIdx.x == 0 && ld_peer_u32(peer_addr(smem_u32(&tmem_slot), (uint32_t)(rank ^ 1))) != tmem) {
    atomicOr(err, 8u);
    stop_flag = 1u;
    remote_stop(stop, (uint32_t)(rank ^ 1));
  }
  cluster_barrier();
  const int ntiles = g.batch * g.tiles_per_matrix;
  const int KB = (g.K + kGemmBK - 1) / kGemmBK;
  const uint32_t leader_full0 = peer_addr(full_bar(0), 0);
  const uint32_t leader_tempty0 = peer_addr(tempty_bar(0), 0);
  auto halt_cluster = [&]() { remote_stop(stop, (uint32_t)(rank ^ 1)); };

  if (warp == 0) {
    if (lane == 0 && *stop == 0u) {
      // ---------------- producer (both CTAs): this CTA's opA and opB rows
      uint32_t it = 0;
      bool halted = false;
      for (int t = cid; t < ntiles && !halted; t += ncid) {
        int b, m0, n0;
        gemm_tile(g, SYM, t, rank, b, m0, n0);
        const int nb0 = n0 + rank * (kGemmBN / 2);  // this CTA's opB rows
        for (int kb = 0; kb < KB; ++kb) {
          const int s = it % kGemmStages;
          const uint32_t ph = (it / kGemmStages) & 1u;
          if (!mbar_wait(empty_bar(s), ph ^ 1u, err, stop)) {
            halted = true;
            halt_cluster();
            break;
          }
          ++it;
          const uint32_t fb = leader_full0 + 8u * s;  // the leader's full barrier
          if (leader) mbar_expect_tx(full_bar(s), 2 * kGemmStageBytes);
          const uint32_t a = s0 + s * kGemmStageBytes, bb = a + kGemmABytes;
          const int k0 = kb * kGemmBK;
          if (AMN) {
            tma3_g2s_pair(a, &tmA, m0, k0, b, fb);
            tma3_g2s_pair(a + 8192u, &tmA, m0 + 64, k0, b, fb);
          } else {
            tma3_g2s_pair(a, &tmA, k0, m0, b, fb);
          }
          if (BMN) {
            tma3_g2s_pair(bb, &tmB, nb0, k0, b, fb);
            tma3_g2s_pair(bb + 8192u, &tmB, nb0 + 64, k0, b, fb);
          } else {
            tma3_g2s_pair(bb, &tmB, k0, nb0, b, fb);
          }
        }
      }
      // the leader sees every copy of both CTAs land; the follower's copies
      // are covered by the leader's wait and the final cluster barrier
      if (leader) {
        const uint64_t deadline = global_ns() + kWaitNs;
        for (int s = 0; s < kGemmStages; ++s) {
          if (it > (uint32_t)s) {
            const uint32_t last = (it - 1 - s) / kGemmStages * kGemmStages + s;
            mbar_drain(full_bar(s), (last / kGemmStages) & 1u, deadline, err);
          }
        }
      }
    }
  } else if (warp == 1) {
    if (lane == 0 && leader && *stop == 0u) {
      // ---------------- MMA issuer (leader only)
      constexpr uint32_t idesc = umma_idesc_bf16(AMN, BMN, 2 * kGemmBM, kGemmBN);
      uint32_t it = 0;
      int lt = 0;
      bool halted = false;
      for (int t = cid; t < ntiles && !halted; t += ncid, ++lt) {
        const int buf = lt & 1;
        const uint32_t tph = ((uint32_t)(lt >> 1) & 1u) ^ 1u;
        if (!mbar_wait_cluster(tempty_bar(buf), tph, err, stop)) {
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
            umma_pair_bf16(d, operand_desc<AMN>(a, kk), operand_desc<BMN>(bb, kk), idesc,
                       (kb | kk) != 0 ? 1u : 0u);
          umma_pair_commit(empty_bar(s), kBoth);  // both CTAs may refill the stage
        }
        if (!halted) umma_pair_commit(tfull_bar(buf), kBoth);
      }
      umma_pair_commit(done_bar, 1);  // this CTA only
      mbar_drain(done_bar, 0u, global_ns() + kWaitNs, err);
    }
  } else {
    // ---------------- epilogue (both CTAs): this CTA's 128 rows
    const int q = warp & 3;
    int lt = 0;
    for (int t = cid; t < ntiles; t += ncid, ++lt) {
      const int buf = lt & 1;
      const uint32_t fph = (uint32_t)(lt >> 1) & 1u;
      const bool ok = __all_sync(0xffffffffu, mbar_wait(tfull_bar(buf), fph, err, stop));
      tc_fence_after();
      if (ok) {
        int b, m0, n0;
        gemm_tile(g, SYM, t, rank, b, m0, n0);
        const int i = m0 + 32 * q + lane;
        const bool row_ok = i < g.M;
        uint16_t* Db = g.D + (int64_t)b * g.sd;
        const uint16_t* Cb = g.beta != 0.0f ? g.C + (int64_t)b * g.sc : nullptr;
#pragma unroll 1
        for (int c = 0; c < kGemmBN / 32; ++c) {
          const int j0 = n0 + 32 * c;
          uint32_t r[32];
          __syncwarp();
          tmem_ld32(tmem + (uint32_t)(buf * kGemmBN + 32 * c) + ((uint32_t)(32 * q) << 16), r);
          if (!row_ok || j0 >= g.N) continue;
          if (SYM && j0 + 31 < i) continue;
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
      if (lane == 0) mbar_arrive_cluster(leader_tempty0 + 8u * buf);
    }
  }
  tc_fence_before();
  __syncthreads();
  cluster_barrier();  // no CTA frees TMEM or leaves while the pair's MMAs or copies may touch it
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc_pair(tmem, kGemmTmemCols);
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

