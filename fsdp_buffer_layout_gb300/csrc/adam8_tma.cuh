// adam8_tma.cuh — the 8-bit AdamW block kernel for contiguous blocks, with a
// TMA (bulk-copy) pipeline. Included by vsf_kernels.cu after adam8.cuh (same
// element math, same results bit for bit).
//
// Work: cluster c takes the units list[starts[c]] .. list[starts[c+1]-1] in
// turn (the host balances the clusters' element counts at upload).
//
// Structure of one CTA: warps 0..W-1 compute, the last warp (W) is the
// producer. The producer streams fixed-size chunks of the CTA's share of
// each block from global memory into a ring of shared-memory slots with
// cp.async.bulk (the Blackwell bulk-copy engine), each slot guarded by a
// "full" mbarrier (transaction bytes) and an "empty" mbarrier (one arrival per
// consumer warp). Per block the sequence is: every phase-1 chunk (gradient and
// codes, kept in L2 with an evict-last hint; two chunks per slot where they
// fit, as a phase-1 chunk needs half a slot), then every phase-2 chunk
// (gradient and codes again, now L2 hits, plus the master). The producer runs
// ahead across phases and blocks as far as the ring allows, so HBM requests
// keep flowing while the consumers wait for the block maxima.
//
// Block maxima: after phase 1 each CTA's consumers reduce their maxima; lane
// r of warp 0 writes the CTA's pair into a slot of cluster rank r with an
// asynchronous distributed-shared-memory store (st.async), whose bytes
// complete a transaction on that CTA's mbarrier; each CTA posts the
// cluster's byte count on its own barrier once per unit, and its warp 0
// waits there. A second barrier of the consumer warps then publishes the
// maxima to the other warps. A CTA that is its own cluster keeps the maxima
// in its shared memory and needs only that second barrier (a cluster-scope
// exchange with itself cost 6% of the kernel on the 1.3B model).
// Slots and barriers alternate between two sets by block parity.
//
// Every wait is bounded, and a timeout is sticky. The first wait of a CTA
// that runs out (2 s) sets bit 1 of the device error word and the CTA's
// shared "stop" flag; from then on every wait of that CTA returns at once.
// The producer issues no further copy. A consumer warp releases a ring slot
// (arrives on its "empty" barrier) only after its wait for that slot's data
// succeeded, so the producer never refills a slot whose copy may still be in
// flight. Consumers still pass every barrier among themselves and still send
// their block maxima to the peers (which therefore never wait for them), but
// skip the arithmetic and the stores of every chunk whose data they did not
// get. The wait for the peers' maxima has a sticky flag of its own and keeps
// waiting after a copy timeout, so every maxima store into a CTA has landed
// before it exits. Before exit the producer waits, under one more 2 s limit
// in all, for every copy it issued, so no CTA leaves while a copy into it is
// pending.
// The results of a launch that set the error bit are undefined; the kernel
// finishes within a few limits instead of one limit per wait.

#include "mbarrier.cuh"

// One shape of the kernel: W consumer warps and one producer warp per CTA,
// chunks of W * 512 elements, and a ring of 200 KB at 16 warps or
// proportionally less for narrower shapes, so that 16 / W CTAs share an SM.
template <int W>
struct TmaShape {
  static constexpr int threads = (W + 1) * 32;
  static constexpr int chunk = tma_chunk_elems(W);
  // rows per chunk of a tile unit (chunk / 256 columns) are taken with a shift
  static_assert((chunk & (chunk - 1)) == 0, "chunk sizes are powers of two");
  static constexpr int ctas_per_sm = kTmaWideWarps / W;
  static constexpr uint32_t ring_bytes = 200u * 1024u / ctas_per_sm;
};

template <typename GT, int W>
struct TmaLayout {
  static constexpr uint32_t chunk = TmaShape<W>::chunk;
  static constexpr uint32_t grad = 0;
  static constexpr uint32_t mq = chunk * sizeof(GT);
  static constexpr uint32_t vq = mq + chunk;
  static constexpr uint32_t master = vq + chunk;
  static constexpr uint32_t slot = master + chunk * 4;  // bytes per slot
  // A phase-1 ring chunk holds no master, so where two chunks' gradient and
  // codes fit in a slot, phase 1 takes chunks in pairs (p1 = 2): the same
  // ring then keeps twice the phase-1 bytes in flight.
  static constexpr int p1 = 2 * chunk * (sizeof(GT) + 2) <= slot ? 2 : 1;
  static constexpr uint32_t grad1 = 0;
  static constexpr uint32_t mq1 = p1 * chunk * sizeof(GT);
  static constexpr uint32_t vq1 = mq1 + p1 * chunk;
  static_assert(vq1 + p1 * chunk <= slot, "phase-1 chunks fit in a slot");
  // ring depth: as many slots as fit in the shape's ring, at least two
  static constexpr uint32_t budget = TmaShape<W>::ring_bytes;
  static constexpr int slots = (budget / slot) < 2 ? 2 : (int)(budget / slot);
  static constexpr uint32_t ring = slot * slots;
  // then: full[slots], empty[slots], maxbar[2] (8 B each), and the block
  // maxima maxima[2][kMaxCluster][kMaxUnitTiles] (float2)
  static constexpr uint32_t bars = ring;
  static constexpr uint32_t maxima = bars + 8 * (2 * slots + 2);
  // +128: the kernel rounds the dynamic shared memory base up to 128 bytes
  static constexpr uint32_t total = maxima + 2 * kMaxCluster * kMaxUnitTiles * 8 + 128;
};

// global -> shared bulk copy completing on `bar`, with an L2 cache policy.
__device__ __forceinline__ void bulk_g2s(uint32_t dst, const void* src, uint32_t bytes,
                                         uint32_t bar, uint64_t pol) {
  asm volatile(
      "cp.async.bulk.shared::cta.global.mbarrier::complete_tx::bytes.L2::cache_hint"
      " [%0], [%1], %2, [%3], %4;" ::"r"(dst),
      "l"(src), "r"(bytes), "r"(bar), "l"(pol)
      : "memory");
}

// 2-D tensor copy (global -> shared) of one box at (x, y), completing on `bar`.
__device__ __forceinline__ void tensor2d_g2s(uint32_t dst, const void* tmap, int x, int y,
                                             uint32_t bar, uint64_t pol) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint"
      " [%0], [%1, {%2, %3}], [%4], %5;" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(tmap)), "r"(x), "r"(y), "r"(bar), "l"(pol)
      : "memory");
}

// Tensor maps of the tile tensors (per array: gradient, m codes, v codes,
// master), passed as a grid constant.
struct TileMaps {
  CUtensorMap m[kMaxTileMaps][4];
  int32_t tensor[kMaxTileMaps];
  int32_t count;
};

// Fetch the line holding *p into this SM's L1 (no register, no wait).
__device__ __forceinline__ void prefetch_l1(const void* p) {
  asm volatile("prefetch.global.L1 [%0];" ::"l"(p));
}

// Asynchronous remote store of a float2 into a peer's shared memory: the
// peer's mbarrier at the offset of local_bar receives the 8 bytes as
// transaction bytes, so the peer sees the data once that phase completes,
// with no release fence on this side.
__device__ __forceinline__ void dsmem_put_async(uint32_t local_slot, uint32_t local_bar,
                                                uint32_t rank, float2 v) {
  uint32_t rs, rb;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(rs) : "r"(local_slot), "r"(rank));
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(rb) : "r"(local_bar), "r"(rank));
  asm volatile(
      "st.async.shared::cluster.mbarrier::complete_tx::bytes.v2.f32 [%0], {%1, %2}, [%3];" ::"r"(rs),
      "f"(v.x), "f"(v.y), "r"(rb)
      : "memory");
}

// One ring chunk of a work unit. Contiguous blocks (one row) are cut into
// CH-element pieces (CH: the shape's chunk); a unit of k tiles into boxes of whole rows of
// W = k * tile_cols elements (a power of two <= 256), which the tensor copy
// packs back to back in the slot.
struct TmaChunk {
  int64_t gstart;  // buffer element of the chunk's first element
  int rows;        // rows in the chunk (1 for a contiguous block)
  int row_len;     // elements per row
  int stride;      // buffer elements between rows
  int row_log2;    // log2(row_len) when rows > 1
  __device__ __forceinline__ int len() const { return rows * row_len; }
  // Buffer element of the chunk's element `i` (packed row-major order).
  __device__ __forceinline__ int64_t at(int i) const {
    return rows == 1 ? gstart + i
                     : gstart + (int64_t)(i >> row_log2) * stride + (i & (row_len - 1));
  }
};

// Unit width: the block's row length times its tiles (1 for contiguous).
__device__ __forceinline__ int tma_width(const QBlock& b, int k) { return b.ncols * k; }
template <int CH>
__device__ __forceinline__ int tma_rows_per_chunk(const QBlock& b, int k) {
  // a tile unit's width is a power of two (k tiles of a power-of-two width,
  // one 256-column copy box): a shift, not a division, in every chunk
  return CH >> (31 - __clz(tma_width(b, k)));
}

// The part of a unit that CTA `crank` of CL owns: chunks [c0, c1). A
// contiguous block is split into CL element ranges [e0, e1) of equal length
// to 16 elements (its length is a multiple of 16, so every range starts on a
// 16-byte boundary of the code arrays), each cut into CH-element chunks from
// its start, the last one short; the CTAs then move the same bytes. A tile
// unit is split by whole chunks of rows.
struct TmaShare {
  int c0, c1;
  int e0, e1;  // element range inside a contiguous block
};

template <int CH>
__device__ __forceinline__ TmaShare tma_share(const QBlock& b, int k, int CL, int crank) {
  // rows per chunk and the cluster size are powers of two: shifts
  const int cl_log2 = 31 - __clz(CL);
  TmaShare sh;
  if (b.nrows == 1) {
    const int64_t n16 = b.ncols >> 4;
    sh.e0 = (int)(((n16 * crank) >> cl_log2) << 4);
    sh.e1 = (int)(((n16 * (crank + 1)) >> cl_log2) << 4);
    sh.c0 = 0;
    sh.c1 = (sh.e1 - sh.e0 + CH - 1) / CH;
  } else {
    const int rpc = tma_rows_per_chunk<CH>(b, k);
    const int nch = (b.nrows + rpc - 1) >> (31 - __clz(rpc));
    const int per = (nch + CL - 1) >> cl_log2;
    sh.c0 = min(nch, crank * per);
    sh.c1 = min(nch, sh.c0 + per);
    sh.e0 = sh.e1 = 0;
  }
  return sh;
}

template <int CH>
__device__ __forceinline__ TmaChunk tma_chunk(const QBlock& b, int k, const TmaShare& sh, int c) {
  TmaChunk ch;
  if (b.nrows == 1) {
    const int e = sh.e0 + c * CH;
    ch.gstart = b.base + e;
    ch.rows = 1;
    ch.row_len = min(CH, sh.e1 - e);
    ch.stride = 0;
    ch.row_log2 = 0;
  } else {
    const int rpc = tma_rows_per_chunk<CH>(b, k);
    const int r0 = c * rpc;
    ch.gstart = b.base + (int64_t)r0 * b.stride;
    ch.rows = min(rpc, b.nrows - r0);
    ch.row_len = tma_width(b, k);
    ch.stride = b.stride;
    ch.row_log2 = 31 - __clz(ch.row_len);
  }
  return ch;
}

template <typename GT, int W>
__global__ void __launch_bounds__(TmaShape<W>::threads, TmaShape<W>::ctas_per_sm) adam_tma_kernel(
    const __grid_constant__ TileMaps maps, const QBlock* __restrict__ qb,
    const int32_t* __restrict__ list, const int32_t* __restrict__ ktab,
    const int32_t* __restrict__ starts,
    const GT* __restrict__ grad, const float* __restrict__ d_factor, float* master, int8_t* mq,
    uint8_t* vq, float* m_scale, float* v_scale, uint16_t* bf, AdamConsts k, unsigned* err) {
  using Lay = TmaLayout<GT, W>;
  constexpr int CH = TmaShape<W>::chunk;
  constexpr int kTmaSlots = Lay::slots;
  extern __shared__ __align__(128) unsigned char smem_raw[];
  // tensor copies want 128-byte aligned destinations: round the base up
  unsigned char* smem = smem_raw + ((128u - (smem_u32(smem_raw) & 127u)) & 127u);
  cg::cluster_group cluster = cg::this_cluster();
  const int CL = (int)cluster.num_blocks();
  const int crank = (int)cluster.block_rank();
  const int cid = blockIdx.x / CL;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const uint32_t s0 = smem_u32(smem);
  auto full_bar = [&](int s) { return s0 + Lay::bars + 8u * s; };
  auto empty_bar = [&](int s) { return s0 + Lay::bars + 8u * (kTmaSlots + s); };
  auto max_bar = [&](int par) { return s0 + Lay::bars + 8u * (2 * kTmaSlots + par); };
  float2* maxima = reinterpret_cast<float2*>(smem + Lay::maxima);
  __shared__ uint32_t stop_flag;  // set by the first wait of this CTA that runs out
  volatile uint32_t* stop = &stop_flag;
  // The maxima exchange keeps its own flag: every CTA sends its maxima for
  // every unit even after its copies stopped, so waiting for the peers'
  // stays bounded, keeps the barrier phases in step and leaves no store in
  // flight towards a CTA that has exited.
  __shared__ uint32_t xstop_flag;
  volatile uint32_t* xstop = &xstop_flag;

  if (tid == 0) {
    stop_flag = 0u;
    xstop_flag = 0u;
    for (int s = 0; s < kTmaSlots; ++s) {
      mbar_init(full_bar(s), 1);
      mbar_init(empty_bar(s), W);
    }
    mbar_init(max_bar(0), 1);  // this CTA's own arrival, posting the peers' bytes
    mbar_init(max_bar(1), 1);
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  cluster.sync();

  if (warp == W) {
    // ---------------- producer warp: lane 0 waits for the slot, posts the
    // byte count and issues the copies (one 1-D bulk copy per array for a
    // contiguous chunk, one 2-D tensor copy per array for a tile chunk).
    if (lane == 0) {
      const uint64_t keep = l2_policy_evict_last();
      const uint64_t drop = l2_policy_evict_first();
      uint32_t p = 0;  // ring positions issued so far
      bool halted = false;
      for (int j = starts[cid]; j < starts[cid + 1] && !halted; ++j) {
        const int q0 = list[j];
        const QBlock b = qb[q0];
        const int kt = ktab[j];
        const TmaShare sh = tma_share<CH>(b, kt, CL, crank);
        const int c0 = sh.c0, c1 = sh.c1;
        // The consumers start the unit by reading its tiles' old scales;
        // fetch those lines into this SM's L1 now, ahead of them. Measured
        // on the wide shape: 1.3B model 3.436 -> 3.362 ms, MoE layer 2.226 ->
        // 2.215; the narrow shape (DSv3 block) ran 0.3% slower with it.
        if constexpr (W == kTmaWideWarps) {
          prefetch_l1(m_scale + q0);
          prefetch_l1(m_scale + q0 + kt - 1);
          prefetch_l1(v_scale + q0);
          prefetch_l1(v_scale + q0 + kt - 1);
        }
        int mi = 0;
        if (b.tx >= 0)
          while (mi + 1 < maps.count && maps.tensor[mi] != b.tensor) ++mi;
        for (int ph = 0; ph < 2 && !halted; ++ph) {
          const int step = ph == 0 ? Lay::p1 : 1;
          for (int c = c0; c < c1; c += step) {
            const int s = p % kTmaSlots;
            const uint32_t round = p / kTmaSlots;
            // ring chunk = chunks c .. c + n - 1 of the share (n = 2 for a
            // phase-1 pair), adjacent in the buffer or boxes packed in order
            const int n = min(step, c1 - c);
            const TmaChunk ch = tma_chunk<CH>(b, kt, sh, c);
            const TmaChunk cl = n == 2 ? tma_chunk<CH>(b, kt, sh, c + 1) : ch;
            const uint32_t len0 = (uint32_t)ch.len();
            const uint32_t len = len0 + (n == 2 ? (uint32_t)cl.len() : 0u);
            // the slot is free once every consumer warp has used its last
            // data; after a timeout anywhere in the CTA, stop issuing
            if ((round > 0 && !mbar_wait(empty_bar(s), (round - 1) & 1, err, stop)) || *stop) {
              halted = true;
              break;
            }
            ++p;
            const uint32_t fb = full_bar(s);
            const int64_t last = cl.gstart + (int64_t)(cl.rows - 1) * cl.stride + cl.row_len;
            if (!in_bounds(k.bd, ch.gstart, last)) {
              mbar_arrive(fb);  // no copy: complete the slot's phase without data
              continue;
            }
            mbar_expect_tx(fb, len * (uint32_t)(sizeof(GT) + 2) + (ph ? len * 4u : 0u));
            const uint32_t slot = s0 + s * Lay::slot;
            const uint32_t og = ph ? Lay::grad : Lay::grad1;
            const uint32_t om = ph ? Lay::mq : Lay::mq1;
            const uint32_t ov = ph ? Lay::vq : Lay::vq1;
            const uint64_t pol = ph == 0 ? keep : drop;
            if (b.tx < 0) {
              const int64_t e = ch.gstart;
              bulk_g2s(slot + og, grad + e, len * sizeof(GT), fb, pol);
              bulk_g2s(slot + om, mq + e, len, fb, pol);
              bulk_g2s(slot + ov, vq + e, len, fb, pol);
              if (ph) bulk_g2s(slot + Lay::master, master + e, len * 4u, fb, drop);
            } else {
              for (int i = 0; i < n; ++i) {
                const int y = b.ty + (c + i) * tma_rows_per_chunk<CH>(b, kt);
                const uint32_t at = i * len0;  // elements before this box in the slot
                tensor2d_g2s(slot + og + at * sizeof(GT), &maps.m[mi][0], b.tx, y, fb, pol);
                tensor2d_g2s(slot + om + at, &maps.m[mi][1], b.tx, y, fb, pol);
                tensor2d_g2s(slot + ov + at, &maps.m[mi][2], b.tx, y, fb, pol);
                if (ph) tensor2d_g2s(slot + Lay::master, &maps.m[mi][3], b.tx, y, fb, drop);
              }
            }
          }
        }
      }
      // Every issued copy has normally been consumed before the consumers
      // finish; wait for the last one of each slot anyway (one limit for all
      // slots together, ignoring the stop flag) so that none is in flight at
      // exit.
      const uint64_t deadline = global_ns() + kWaitNs;
      for (int s = 0; s < kTmaSlots; ++s) {
        if (p > (uint32_t)s) {
          const uint32_t last = (p - 1 - s) / kTmaSlots * kTmaSlots + s;  // last position in slot s
          mbar_drain(full_bar(s), (last / kTmaSlots) & 1, deadline, err);
        }
      }
    }
  } else {
    // ---------------- consumers: thread `tid` owns groups tid, tid + 32*W, ...
    Consts2 c;
    c.b1 = f2(k.b1);
    c.omb1 = f2(k.omb1);
    c.b2 = f2(k.b2);
    c.omb2 = f2(k.omb2);
    c.eps_hat = f2(k.eps_hat);
    c.decay = f2(k.decay);
    c.alpha = f2(k.alpha);
    c.factor = f2(*d_factor);
    const uint64_t drop = l2_policy_evict_first();
    __shared__ float red[2][2][W][kMaxUnitTiles];
    uint32_t p = 0;
    int nb = 0;  // units done by this CTA
    for (int j = starts[cid]; j < starts[cid + 1]; ++j, ++nb) {
      const int q0 = list[j];
      const QBlock b = qb[q0];
      const int kt = ktab[j];
      // This thread's groups always sit in the same column group of a row, so
      // in one tile of the unit: tt (0 for a contiguous block).
      const int gpr = b.nrows == 1 ? 32 : tma_width(b, kt) >> 3;  // groups per row (<= 32)
      const int gpt = b.nrows == 1 ? 32 : b.ncols >> 3;           // groups per tile
      const int gpt_log2 = 31 - __clz(gpt);  // gpr and gpt are powers of two
      const int tt = b.nrows == 1 ? 0 : (tid & (gpr - 1)) >> gpt_log2;
      const int q = q0 + tt;
      c.dm = f2(__fdiv_rn(m_scale[q], 127.0f));
      c.dv = f2(__fdiv_rn(v_scale[q], 255.0f));
      const TmaShare sh = tma_share<CH>(b, kt, CL, crank);
      const int c0 = sh.c0, c1 = sh.c1;
      const int par = nb & 1;
      // the block maxima of every CTA of the cluster (8 bytes per tile) will
      // land on this barrier
      if (CL > 1 && tid == 0) mbar_expect_tx(max_bar(par), (uint32_t)(CL * kt * 8));

      // phase 1: maxima of the new moments
      float mx = 0.0f, vx = 0.0f;
      for (int ci = c0; ci < c1; ci += Lay::p1, ++p) {
        const int s = p % kTmaSlots;
        // warp-uniform: the chunk is used (and its slot released) only if
        // every lane saw the data arrive
        const bool got = __all_sync(0xffffffffu, mbar_wait(full_bar(s), (p / kTmaSlots) & 1, err, stop));
        if (!got) continue;
        int len = tma_chunk<CH>(b, kt, sh, ci).len();
        if (Lay::p1 == 2 && ci + 1 < c1) len += tma_chunk<CH>(b, kt, sh, ci + 1).len();
        const unsigned char* sl = smem + s * Lay::slot;
#pragma unroll
        for (int gi = 0; gi < Lay::p1 * kTmaGroups; ++gi) {
          const int g = tid + gi * W * 32;
          if (g * 8 < len) {
            Raw r;
            r.g0 = *reinterpret_cast<const uint4*>(sl + Lay::grad1 + g * 8 * sizeof(GT));
            if constexpr (sizeof(GT) == 4)
              r.g1 = *reinterpret_cast<const uint4*>(sl + Lay::grad1 + g * 32 + 16);
            r.cm = *reinterpret_cast<const uint2*>(sl + Lay::mq1 + g * 8);
            r.cv = *reinterpret_cast<const uint2*>(sl + Lay::vq1 + g * 8);
            phase1_group<GT>(c, r, mx, vx);
          }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(empty_bar(s));
      }
      // Per-tile warp maxima: the lanes of one tile are runs of gpt lanes
      // that repeat every gpr lanes.
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) {
        if (o < gpt || o >= gpr) {
          mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
          vx = fmaxf(vx, __shfl_xor_sync(0xffffffffu, vx, o));
        }
      }
      if (lane < gpr && (lane & (gpt - 1)) == 0) {
        red[par][0][warp][lane >> gpt_log2] = mx;
        red[par][1][warp][lane >> gpt_log2] = vx;
      }
      asm volatile("bar.sync 1, %0;" ::"r"(W * 32) : "memory");
      if (warp == 0) {
        // the CTA's maxima, one warp entry per lane; lane r then sends them
        // to cluster rank r
        for (int t = 0; t < kt; ++t) {
          float bm = lane < W ? red[par][0][lane][t] : 0.0f;
          float bv = lane < W ? red[par][1][lane][t] : 0.0f;
          bm = fmaxf(bm, 0.0f);
          bv = fmaxf(bv, 0.0f);
#pragma unroll
          for (int o = 16; o > 0; o >>= 1) {
            bm = fmaxf(bm, __shfl_xor_sync(0xffffffffu, bm, o));
            bv = fmaxf(bv, __shfl_xor_sync(0xffffffffu, bv, o));
          }
          if (CL == 1) {
            if (lane == 0) maxima[(par * kMaxCluster) * kMaxUnitTiles + t] = make_float2(bm, bv);
          } else if (lane < CL) {
            dsmem_put_async(smem_u32(&maxima[(par * kMaxCluster + crank) * kMaxUnitTiles + t]),
                            max_bar(par), lane, make_float2(bm, bv));
          }
        }
      }
      // A CTA on its own keeps the maxima in its shared memory. In a cluster,
      // warp 0 waits until every CTA's maxima have landed here; either way a
      // second barrier of the consumer warps then publishes them to the
      // other warps.
      if (CL > 1 && warp == 0) mbar_wait_cluster(max_bar(par), (nb >> 1) & 1, err, xstop);
      asm volatile("bar.sync 1, %0;" ::"r"(W * 32) : "memory");
      float sm = 0.0f, sv = 0.0f;
      for (int rk = 0; rk < CL; ++rk) {
        const float2 v = maxima[(par * kMaxCluster + rk) * kMaxUnitTiles + tt];
        sm = fmaxf(sm, v.x);
        sv = fmaxf(sv, v.y);
      }
      c.im = f2(sm > 0.0f ? __fdiv_rn(127.0f, sm) : 0.0f);
      c.iv = f2(sv > 0.0f ? __fdiv_rn(255.0f, sv) : 0.0f);
      if (crank == 0 && tid < kt * gpt && (tid & (gpt - 1)) == 0 && *stop == 0u) {  // one thread per tile
        m_scale[q] = sm;
        v_scale[q] = sv;
      }

      // phase 2: update, requantise, write
      for (int ci = c0; ci < c1; ++ci, ++p) {
        const int s = p % kTmaSlots;
        const bool got = __all_sync(0xffffffffu, mbar_wait(full_bar(s), (p / kTmaSlots) & 1, err, stop));
        if (!got) continue;
        const TmaChunk ch = tma_chunk<CH>(b, kt, sh, ci);
        const int len = ch.len();
        const unsigned char* sl = smem + s * Lay::slot;
#pragma unroll
        for (int gi = 0; gi < kTmaGroups; ++gi) {
          const int g = tid + gi * W * 32;
          if (g * 8 < len) {
            Raw r;
            r.g0 = *reinterpret_cast<const uint4*>(sl + Lay::grad + g * 8 * sizeof(GT));
            if constexpr (sizeof(GT) == 4)
              r.g1 = *reinterpret_cast<const uint4*>(sl + Lay::grad + g * 32 + 16);
            r.cm = *reinterpret_cast<const uint2*>(sl + Lay::mq + g * 8);
            r.cv = *reinterpret_cast<const uint2*>(sl + Lay::vq + g * 8);
            const uint4 pa = *reinterpret_cast<const uint4*>(sl + Lay::master + g * 32);
            const uint4 pb = *reinterpret_cast<const uint4*>(sl + Lay::master + g * 32 + 16);
            uint4 o0, o1, ob;
            uint2 ocm, ocv;
            phase2_group<GT>(c, r, pa, pb, o0, o1, ob, ocm, ocv);
            const int64_t e = ch.at(g * 8);
            if (!in_bounds(k.bd, e, e + 8)) continue;
            st_v4(master + e, o0, drop);
            st_v4(master + e + 4, o1, drop);
            st_v4(bf + e, ob, drop);
            st_v2(mq + e, ocm, drop);
            st_v2(vq + e, ocv, drop);
          }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(empty_bar(s));
      }
    }
  }
  __syncwarp();
  cluster.sync();  // no CTA leaves while a peer may still write into it
  // When launched alongside the element-chunk kernel (programmatic
  // serialization), finish only after it, so that later launches on the
  // stream see both kernels' writes. Returns at once otherwise.
  asm volatile("griddepcontrol.wait;" ::: "memory");
}

// Self-test of the bounded wait: one CTA waits, four times in a row, on
// barriers that no one arrives on. The first wait must give up after
// limit_ns and set bit 1 of err[0]; the timeout is sticky, so the other three
// return at once. err[1] receives the elapsed time of the four waits in
// microseconds (about one limit, not four).
__global__ void wait_selftest_kernel(unsigned* err, uint64_t limit_ns) {
  __shared__ __align__(8) uint64_t bar[4];
  __shared__ uint32_t stop_flag;
  if (threadIdx.x == 0) {
    stop_flag = 0u;
    for (int i = 0; i < 4; ++i) mbar_init(smem_u32(&bar[i]), 1);
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    const uint64_t t0 = global_ns();
    for (int i = 0; i < 4; ++i) mbar_wait(smem_u32(&bar[i]), 0, err, &stop_flag, limit_ns);
    err[1] = (unsigned)((global_ns() - t0) / 1000u);
  }
}
