// adam8.cuh — block-wise 8-bit AdamW kernels of libvsf (sm_103a).
// Included by vsf_kernels.cu inside namespace vsf::{anonymous}.
//
// Method: "veScale-FSDP: Flexible and High-Performance FSDP at Scale (MLSys
// 2026)" summary page › 结构感知训练 case study › 8-bit Adam: quantisation
// blocks are never split across ranks, so every block's scale is computed
// from data of one rank only. The quantiser and the op order are readings
// (the pages define neither):
//   g  = factor * grad
//   m  = b1 * m' + (1 - b1) * g,      m' = code_m * (m_scale / 127)
//   v  = b2 * v' + (1 - b2) * (g*g),  v' = code_v * (v_scale / 255)
//   p  = p * (1 - lr*wd)
//   p  = p - alpha_t * (m / (sqrt(v) + eps_hat))
//        alpha_t = lr sqrt(1-b2^t) / (1-b1^t), eps_hat = eps sqrt(1-b2^t)
//        (the efficient form of the bias-corrected update given at the end
//        of section 2 of Kingma & Ba's Adam paper)
//   bf16 copy = round-to-nearest-even(p)
//   new m_scale = max |m|, new v_scale = max v over the block;
//   codes = round-half-even(m * (127 / m_scale)) saturated to [-127, 127]
//           and round-half-even(v * (255 / v_scale)) saturated to [0, 255],
//           NaN -> 0.
// Every fp32 operation is an explicit round-to-nearest operation, scalar
// (__fmul_rn, __fadd_rn, __fdiv_rn, __fsqrt_rn) or a packed multiply
// (mul.rn.f32x2 in inline PTX, which rounds each component like the scalar
// form), and the library is compiled with -fmad=false: no multiply and add
// are ever contracted into one FMA, so the results equal a plain C
// implementation of the same sequence bit for bit.
//
// Work decomposition (one HBM pass): a quantisation block needs its new
// absmax before any code can be written. One thread-block cluster takes one
// block at a time; each CTA of the cluster owns an equal share. Phase 1 reads
// gradient and codes (4 B per element for bf16 gradients, with an L2
// evict-last hint), computes the new moments and their maxima; the CTAs of a
// cluster swap maxima through distributed shared memory (a CTA on its own
// keeps them in its shared memory); phase 2
// re-reads the same share (an L2 hit: at most clusters x block bytes were
// read in between), reads the master once, and writes master, bf16 copy and
// codes with evict-first hints. HBM sees every byte once.

struct AdamConsts {
  float b1, omb1, b2, omb2, eps_hat, decay, alpha;
  Bounds bd;  // index checks of the debug build
};

// ---------------------------------------------------------------- memory ops

__device__ __forceinline__ uint64_t l2_policy_evict_last() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(p));
  return p;
}
__device__ __forceinline__ uint64_t l2_policy_evict_first() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
  return p;
}
__device__ __forceinline__ uint4 ld_v4(const void* ptr, uint64_t pol) {
  uint4 r;
  asm volatile("ld.global.L2::cache_hint.v4.u32 {%0,%1,%2,%3}, [%4], %5;"
               : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
               : "l"(ptr), "l"(pol));
  return r;
}
__device__ __forceinline__ uint2 ld_v2(const void* ptr, uint64_t pol) {
  uint2 r;
  asm volatile("ld.global.L2::cache_hint.v2.u32 {%0,%1}, [%2], %3;"
               : "=r"(r.x), "=r"(r.y)
               : "l"(ptr), "l"(pol));
  return r;
}
__device__ __forceinline__ void st_v4(void* ptr, uint4 v, uint64_t pol) {
  asm volatile("st.global.L2::cache_hint.v4.u32 [%0], {%1,%2,%3,%4}, %5;" ::"l"(ptr), "r"(v.x),
               "r"(v.y), "r"(v.z), "r"(v.w), "l"(pol)
               : "memory");
}
__device__ __forceinline__ void st_v2(void* ptr, uint2 v, uint64_t pol) {
  asm volatile("st.global.L2::cache_hint.v2.u32 [%0], {%1,%2}, %3;" ::"l"(ptr), "r"(v.x),
               "r"(v.y), "l"(pol)
               : "memory");
}

// Bulk prefetch of [begin, end) into L2 (one instruction per range, no
// registers held). The range is shrunk to whole 16-byte units inside it, as
// the bulk copy engine requires, so no byte outside [begin, end) is touched.
__device__ __forceinline__ void prefetch_l2(const void* begin, const void* end) {
  const uintptr_t b = (reinterpret_cast<uintptr_t>(begin) + 15) & ~uintptr_t(15);
  const uintptr_t e = reinterpret_cast<uintptr_t>(end) & ~uintptr_t(15);
  if (e <= b) return;
  asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(b), "r"((uint32_t)(e - b))
               : "memory");
}

// ---------------------------------------------------------------- element math

__device__ __forceinline__ float2 f2(float a) { return make_float2(a, a); }

// Packed fp32x2 multiply with an explicit round-to-nearest modifier: each
// component rounds exactly like mul.rn.f32. Additions stay scalar
// (__fadd_rn). Measured on 2^20 random operands: a packed add alone
// (add.rn.f32x2) matches the scalar add on every operand, but after a packed
// multiply the device compiler fuses the two into one rounding in 23% of
// cases, -fmad=false notwithstanding. An fma by a run-time 1.0 instead keeps
// both roundings (and parity), but ran 0.2-1.4% slower than scalar adds.
__device__ __forceinline__ float2 mul2(float2 a, float2 b) {
  float2 d;
  asm("{\n .reg .b64 ra, rb, rd;\n mov.b64 ra, {%2, %3};\n mov.b64 rb, {%4, %5};\n"
      " mul.rn.f32x2 rd, ra, rb;\n mov.b64 {%0, %1}, rd;\n}"
      : "=f"(d.x), "=f"(d.y)
      : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y));
  return d;
}

// Codes to exact floats: 2^23 + byte has the byte in its low mantissa bits,
// and subtracting 2^23 (2^23 + 128 for the offset signed codes) is exact, so
// the packed add here rounds nothing (and no multiply feeds it).
__device__ __forceinline__ float2 u8pair_to_f2(uint32_t word, int first) {
  const float2 x = make_float2(__uint_as_float(__byte_perm(word, 0x4B000000u, 0x7540u | first)),
                               __uint_as_float(__byte_perm(word, 0x4B000000u, 0x7541u | first)));
  return __fadd2_rn(x, f2(-8388608.0f));
}
__device__ __forceinline__ float2 s8pair_to_f2(uint32_t word_xor80, int first) {
  const float2 x =
      make_float2(__uint_as_float(__byte_perm(word_xor80, 0x4B000000u, 0x7540u | first)),
                  __uint_as_float(__byte_perm(word_xor80, 0x4B000000u, 0x7541u | first)));
  return __fadd2_rn(x, f2(-8388736.0f));  // 2^23 + 128
}

// m code: round-half-even, saturated to the symmetric range [-127, 127]
// (never -128). The lower clamp comes first and keeps a NaN a NaN
// (max.NaN), which the conversion then turns into 0. It matters when a
// block's scale is so small that 127 / scale overflows to infinity.
// Both conversions leave the code in byte 0 of the word (the upper bytes
// extend it); every caller takes byte 0 only (pack4, or a cast to an 8-bit
// type), so no mask is spent on them.
__device__ __forceinline__ uint32_t cvt_sat_s8(float x) {
  float y;
  asm("max.NaN.f32 %0, %1, 0fC2FE0000;" : "=f"(y) : "f"(x));  // max(x, -127)
  uint32_t r;
  asm("cvt.rni.sat.s8.f32 %0, %1;" : "=r"(r) : "f"(y));
  return r;
}
__device__ __forceinline__ uint32_t cvt_sat_u8(float x) {
  uint32_t r;
  asm("cvt.rni.sat.u8.f32 %0, %1;" : "=r"(r) : "f"(x));
  return r;
}
// Bytes 0 of a, b, c, d, in that order from the low byte.
__device__ __forceinline__ uint32_t pack4(uint32_t a, uint32_t b, uint32_t c, uint32_t d) {
  return __byte_perm(__byte_perm(a, b, 0x0040u), __byte_perm(c, d, 0x0040u), 0x5410u);
}

__device__ __forceinline__ uint32_t bf16x2_bits(float lo, float hi) {
  const __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<const uint32_t*>(&h);
}
__device__ __forceinline__ uint32_t bf16_bits(float x) { return bf16x2_bits(x, 0.0f) & 0xffffu; }

struct Consts2 {
  float2 b1, omb1, b2, omb2, eps_hat, decay, alpha;
  float2 factor, dm, dv, im, iv;
};

// Moments of two elements (packed, bit-identical to the scalar sequence).
__device__ __forceinline__ float2 add2(float2 a, float2 b) {
  return make_float2(__fadd_rn(a.x, b.x), __fadd_rn(a.y, b.y));
}

// Moments of two elements (packed multiplies, scalar adds; bit-identical to
// the scalar sequence).
__device__ __forceinline__ void moments2(const Consts2& c, float2 gin, float2 qm, float2 qv,
                                         float2& m, float2& v) {
  const float2 g = mul2(c.factor, gin);
  const float2 mp = mul2(qm, c.dm);
  const float2 vp = mul2(qv, c.dv);
  m = add2(mul2(c.b1, mp), mul2(c.omb1, g));
  v = add2(mul2(c.b2, vp), mul2(c.omb2, mul2(g, g)));
}

__device__ __forceinline__ float2 update2(const Consts2& c, float2 p, float2 m, float2 v) {
  p = mul2(p, c.decay);
  const float2 den = add2(make_float2(__fsqrt_rn(v.x), __fsqrt_rn(v.y)), c.eps_hat);
  const float2 q = make_float2(__fdiv_rn(m.x, den.x), __fdiv_rn(m.y, den.y));
  const float2 s = mul2(c.alpha, q);
  return make_float2(__fsub_rn(p.x, s.x), __fsub_rn(p.y, s.y));
}

// Scalar twins for ragged groups (same operations, same order).
__device__ __forceinline__ void moments1(const Consts2& c, float gin, float qm, float qv, float& m,
                                         float& v) {
  const float g = __fmul_rn(c.factor.x, gin);
  const float mp = __fmul_rn(qm, c.dm.x);
  const float vp = __fmul_rn(qv, c.dv.x);
  m = __fadd_rn(__fmul_rn(c.b1.x, mp), __fmul_rn(c.omb1.x, g));
  v = __fadd_rn(__fmul_rn(c.b2.x, vp), __fmul_rn(c.omb2.x, __fmul_rn(g, g)));
}
__device__ __forceinline__ float update1(const Consts2& c, float p, float m, float v) {
  p = __fmul_rn(p, c.decay.x);
  const float den = __fadd_rn(__fsqrt_rn(v), c.eps_hat.x);
  return __fsub_rn(p, __fmul_rn(c.alpha.x, __fdiv_rn(m, den)));
}

template <typename GT>
__device__ __forceinline__ float2 grad_pair(const uint4& gr0, const uint4& gr1, int j);

// bf16 gradients: one uint4 holds 8 elements, pair j is its word j.
template <>
__device__ __forceinline__ float2 grad_pair<uint16_t>(const uint4& gr, const uint4&, int j) {
  const uint32_t w = j == 0 ? gr.x : j == 1 ? gr.y : j == 2 ? gr.z : gr.w;
  return make_float2(__uint_as_float(w << 16), __uint_as_float(w & 0xffff0000u));
}
// fp32 gradients: two uint4 hold 8 elements.
template <>
__device__ __forceinline__ float2 grad_pair<float>(const uint4& a, const uint4& b, int j) {
  const uint4& r = j < 2 ? a : b;
  return (j & 1) ? make_float2(__uint_as_float(r.z), __uint_as_float(r.w))
                 : make_float2(__uint_as_float(r.x), __uint_as_float(r.y));
}

// Raw inputs of one full 8-element group.
struct Raw {
  uint4 g0, g1;  // gradient (g1 used for fp32 only)
  uint2 cm, cv;  // codes
};

template <typename GT>
__device__ __forceinline__ void load_raw(const GT* grad, const int8_t* mq, const uint8_t* vq,
                                         int64_t e, uint64_t pol, Raw& r) {
  r.g0 = ld_v4(grad + e, pol);
  if constexpr (sizeof(GT) == 4) r.g1 = ld_v4(grad + e + 4, pol);
  r.cm = ld_v2(mq + e, pol);
  r.cv = ld_v2(vq + e, pol);
}

template <typename GT>
__device__ __forceinline__ void phase1_group(const Consts2& c, const Raw& r, float& mx, float& vx) {
  const uint32_t cmx = r.cm.x ^ 0x80808080u, cmy = r.cm.y ^ 0x80808080u;
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    const uint32_t wm = j < 2 ? cmx : cmy, wv = j < 2 ? r.cv.x : r.cv.y;
    float2 m, v;
    moments2(c, grad_pair<GT>(r.g0, r.g1, j), s8pair_to_f2(wm, 2 * (j & 1)),
             u8pair_to_f2(wv, 2 * (j & 1)), m, v);
    mx = fmaxf(mx, fmaxf(fabsf(m.x), fabsf(m.y)));
    vx = fmaxf(vx, fmaxf(v.x, v.y));
  }
}

template <typename GT>
__device__ __forceinline__ void phase2_group(const Consts2& c, const Raw& r, const uint4& pa,
                                             const uint4& pb, uint4& p_out0, uint4& p_out1,
                                             uint4& bf_out, uint2& cm_out, uint2& cv_out) {
  const uint32_t cmx = r.cm.x ^ 0x80808080u, cmy = r.cm.y ^ 0x80808080u;
  uint32_t qm[8], qv[8], hb[4];
  float po[8];
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    const uint32_t wm = j < 2 ? cmx : cmy, wv = j < 2 ? r.cv.x : r.cv.y;
    float2 m, v;
    moments2(c, grad_pair<GT>(r.g0, r.g1, j), s8pair_to_f2(wm, 2 * (j & 1)),
             u8pair_to_f2(wv, 2 * (j & 1)), m, v);
    const uint4& pr = j < 2 ? pa : pb;
    const float2 p = (j & 1) ? make_float2(__uint_as_float(pr.z), __uint_as_float(pr.w))
                             : make_float2(__uint_as_float(pr.x), __uint_as_float(pr.y));
    const float2 pn = update2(c, p, m, v);
    po[2 * j] = pn.x;
    po[2 * j + 1] = pn.y;
    hb[j] = bf16x2_bits(pn.x, pn.y);
    const float2 xm = mul2(m, c.im), xv = mul2(v, c.iv);
    qm[2 * j] = cvt_sat_s8(xm.x);
    qm[2 * j + 1] = cvt_sat_s8(xm.y);
    qv[2 * j] = cvt_sat_u8(xv.x);
    qv[2 * j + 1] = cvt_sat_u8(xv.y);
  }
  p_out0 = make_uint4(__float_as_uint(po[0]), __float_as_uint(po[1]), __float_as_uint(po[2]),
                      __float_as_uint(po[3]));
  p_out1 = make_uint4(__float_as_uint(po[4]), __float_as_uint(po[5]), __float_as_uint(po[6]),
                      __float_as_uint(po[7]));
  bf_out = make_uint4(hb[0], hb[1], hb[2], hb[3]);
  cm_out = make_uint2(pack4(qm[0], qm[1], qm[2], qm[3]), pack4(qm[4], qm[5], qm[6], qm[7]));
  cv_out = make_uint2(pack4(qv[0], qv[1], qv[2], qv[3]), pack4(qv[4], qv[5], qv[6], qv[7]));
}

// Ragged group (fewer than 8 elements, or not 16-byte aligned): scalar.
template <typename GT>
__device__ __forceinline__ void phase1_scalar(const Consts2& c, const GT* grad, const int8_t* mq,
                                              const uint8_t* vq, int64_t e, int cnt, float& mx,
                                              float& vx) {
  for (int i = 0; i < cnt; ++i) {
    float m, v;
    moments1(c, elem_f32(grad[e + i]), (float)mq[e + i], (float)vq[e + i], m, v);
    mx = fmaxf(mx, fabsf(m));
    vx = fmaxf(vx, v);
  }
}
template <typename GT>
__device__ __forceinline__ void phase2_scalar(const Consts2& c, const GT* grad, int8_t* mq,
                                              uint8_t* vq, float* master, uint16_t* bf, int64_t e,
                                              int cnt) {
  for (int i = 0; i < cnt; ++i) {
    float m, v;
    moments1(c, elem_f32(grad[e + i]), (float)mq[e + i], (float)vq[e + i], m, v);
    const float p = update1(c, master[e + i], m, v);
    master[e + i] = p;
    bf[e + i] = (uint16_t)bf16_bits(p);
    mq[e + i] = (int8_t)cvt_sat_s8(__fmul_rn(m, c.im.x));
    vq[e + i] = (uint8_t)cvt_sat_u8(__fmul_rn(v, c.iv.x));
  }
}

// Where group `i` of this CTA's share starts, and how many elements it has.
struct Share {
  int64_t base;    // buffer element of the block's first element
  int64_t first;   // first group (contiguous) or first row (tiled)
  int ngroups;     // groups in this share
  int vpr_log2;    // tiled: log2(groups per row); -1 contiguous; -2 other rows
  int stride;      // tiled: elements between rows
  int ncols;       // contiguous: block length; tiled: row length
  bool vec;        // 16-byte vector path allowed
  __device__ __forceinline__ void locate(int i, int64_t& e, int& cnt) const {
    if (vpr_log2 < 0) {
      const int64_t off = (first + i) * 8;
      e = base + off;
      cnt = (int)min64(8, (int64_t)ncols - off);
    } else {
      const int r = i >> vpr_log2, v = i & ((1 << vpr_log2) - 1);
      e = base + (first + r) * (int64_t)stride + v * 8;
      cnt = min(8, ncols - v * 8);
    }
  }
  // L2 prefetch of groups [g0, g1) of this share for the arrays given
  // (element size in bytes; null arrays skipped): thread 0 issues one bulk
  // prefetch per array. Only contiguous shares are prefetched; a tile's rows
  // would need one prefetch each, which costs more than it hides.
  __device__ __forceinline__ void prefetch(int g0, int g1, const void* a, int ea, const void* b,
                                           int eb, const void* c, int ec, int tid,
                                           int /*nthreads*/) const {
    g1 = min(g1, ngroups);
    if (g0 >= g1) return;
    auto one = [&](int64_t e0, int64_t e1) {
      if (a) prefetch_l2((const char*)a + e0 * ea, (const char*)a + e1 * ea);
      if (b) prefetch_l2((const char*)b + e0 * eb, (const char*)b + e1 * eb);
      if (c) prefetch_l2((const char*)c + e0 * ec, (const char*)c + e1 * ec);
    };
    if (vpr_log2 == -1) {
      if (tid == 0)
        one(base + (first + g0) * 8, base + min64((first + g1) * 8, (int64_t)ncols));
    }
  }
};

// The share of CTA `crank` of a CL-CTA cluster in block b.
__device__ __forceinline__ Share make_share(const QBlock& b, int CL, int crank) {
  Share sh;
  sh.base = b.base;
  sh.ncols = b.ncols;
  sh.stride = b.stride;
  const int vpr = (b.ncols + 7) >> 3;
  sh.vec = (b.base & 7) == 0;
  if (b.nrows == 1) {
    const int per = (vpr + CL - 1) / CL;
    const int g0 = min(vpr, crank * per);
    sh.first = g0;
    sh.ngroups = min(vpr, g0 + per) - g0;
    sh.vpr_log2 = -1;
  } else {
    const int per = (b.nrows + CL - 1) / CL;
    const int r0 = min(b.nrows, crank * per);
    const int nr = min(b.nrows, r0 + per) - r0;
    sh.first = r0;
    sh.vec = sh.vec && (b.stride & 7) == 0;
    const int lg = 31 - __clz(vpr);
    if ((1 << lg) == vpr) {
      sh.vpr_log2 = lg;
      sh.ngroups = nr * vpr;
    } else {
      sh.vpr_log2 = -2;  // rows whose group count is not a power of two: row by row
      sh.ngroups = nr;
    }
  }
  return sh;
}

// Row / tile blocks, one cluster per block. kThreads threads per CTA; phase 1
// keeps kU1 groups of loads in flight per thread, phase 2 kU2.
template <typename GT, int kThreads, int kMinBlocks, int kU1, int kU2>
__global__ void __launch_bounds__(kThreads, kMinBlocks) adam_block_kernel(
    const QBlock* __restrict__ qb, const int32_t* __restrict__ list, int nlist, int nclusters,
    const GT* __restrict__ grad, const float* __restrict__ d_factor, float* master, int8_t* mq,
    uint8_t* vq, float* m_scale, float* v_scale, uint16_t* bf, AdamConsts k) {
  cg::cluster_group cluster = cg::this_cluster();
  const int CL = (int)cluster.num_blocks();
  const int crank = (int)cluster.block_rank();
  const int cid = blockIdx.x / CL;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  constexpr int kWarps = kThreads / 32;
  __shared__ float red[2][2][kWarps];
  __shared__ float2 slots[2][kMaxCluster];
  const uint64_t keep = l2_policy_evict_last();
  const uint64_t drop = l2_policy_evict_first();

  Consts2 c;
  c.b1 = f2(k.b1);
  c.omb1 = f2(k.omb1);
  c.b2 = f2(k.b2);
  c.omb2 = f2(k.omb2);
  c.eps_hat = f2(k.eps_hat);
  c.decay = f2(k.decay);
  c.alpha = f2(k.alpha);
  c.factor = f2(*d_factor);

  int par = 0;
  for (int j = cid; j < nlist; j += nclusters, par ^= 1) {
    const int q = list[j];
    const QBlock b = qb[q];
    // the same answer in every CTA of the cluster: all skip together
    if (!in_bounds(k.bd, b.base, b.base + (int64_t)(b.nrows - 1) * b.stride + b.ncols)) continue;
    c.dm = f2(__fdiv_rn(m_scale[q], 127.0f));
    c.dv = f2(__fdiv_rn(v_scale[q], 255.0f));

    const Share sh = make_share(b, CL, crank);
    const bool vec = sh.vec;
    const int vpr = (b.ncols + 7) >> 3;
    constexpr int kStep1 = kThreads * kU1, kStep2 = kThreads * kU2;
    if (j == cid) sh.prefetch(0, 2 * kStep1, grad, sizeof(GT), mq, 1, vq, 1, tid, kThreads);

    // ---- phase 1
    float mx = 0.0f, vx = 0.0f;
    if (sh.vpr_log2 >= -1) {
      for (int i0 = tid; i0 < sh.ngroups; i0 += kStep1) {
        const int it0 = i0 - tid;
        sh.prefetch(it0 + 2 * kStep1, it0 + 3 * kStep1, grad, sizeof(GT), mq, 1, vq, 1, tid,
                    kThreads);
        Raw r[kU1];
        bool full[kU1];
        int64_t e[kU1];
        int cnt[kU1];
#pragma unroll
        for (int u = 0; u < kU1; ++u) {
          const int i = i0 + u * kThreads;
          full[u] = false;
          if (i < sh.ngroups) {
            sh.locate(i, e[u], cnt[u]);
            full[u] = vec && cnt[u] == 8;
            if (full[u]) load_raw<GT>(grad, mq, vq, e[u], keep, r[u]);
          }
        }
#pragma unroll
        for (int u = 0; u < kU1; ++u) {
          const int i = i0 + u * kThreads;
          if (full[u])
            phase1_group<GT>(c, r[u], mx, vx);
          else if (i < sh.ngroups)
            phase1_scalar<GT>(c, grad, mq, vq, e[u], cnt[u], mx, vx);
        }
      }
    } else {
      for (int rr = warp; rr < sh.ngroups; rr += kWarps) {
        const int64_t row = sh.base + (sh.first + rr) * (int64_t)sh.stride;
        for (int v = lane; v < vpr; v += 32)
          phase1_scalar<GT>(c, grad, mq, vq, row + v * 8, min(8, sh.ncols - v * 8), mx, vx);
      }
    }

    // master of the first phase-2 iterations, fetched across the barrier
    sh.prefetch(0, 2 * kStep2, master, 4, nullptr, 0, nullptr, 0, tid, kThreads);

    // ---- block maxima: warp, CTA, then cluster through distributed smem
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
      for (int rk = 0; rk < CL; ++rk)
        *cluster.map_shared_rank(&slots[par][crank], rk) = make_float2(bm, bv);
    }
    cluster.sync();
    float sm = 0.0f, sv = 0.0f;
    for (int rk = 0; rk < CL; ++rk) {
      sm = fmaxf(sm, slots[par][rk].x);
      sv = fmaxf(sv, slots[par][rk].y);
    }
    c.im = f2(sm > 0.0f ? __fdiv_rn(127.0f, sm) : 0.0f);
    c.iv = f2(sv > 0.0f ? __fdiv_rn(255.0f, sv) : 0.0f);
    if (crank == 0 && tid == 0) {
      m_scale[q] = sm;
      v_scale[q] = sv;
    }

    // ---- phase 2 (and the next block's first phase-1 data)
    if (j + nclusters < nlist) {
      const Share nx = make_share(qb[list[j + nclusters]], CL, crank);
      nx.prefetch(0, 2 * kStep1, grad, sizeof(GT), mq, 1, vq, 1, tid, kThreads);
    }
    if (sh.vpr_log2 >= -1) {
      for (int i0 = tid; i0 < sh.ngroups; i0 += kStep2) {
        const int it0 = i0 - tid;
        sh.prefetch(it0 + 2 * kStep2, it0 + 3 * kStep2, master, 4, nullptr, 0, nullptr, 0, tid,
                    kThreads);
        Raw r[kU2];
        uint4 pa[kU2], pb[kU2];
        bool full[kU2];
        int64_t e[kU2];
        int cnt[kU2];
#pragma unroll
        for (int u = 0; u < kU2; ++u) {
          const int i = i0 + u * kThreads;
          full[u] = false;
          if (i < sh.ngroups) {
            sh.locate(i, e[u], cnt[u]);
            full[u] = vec && cnt[u] == 8;
            if (full[u]) {
              load_raw<GT>(grad, mq, vq, e[u], drop, r[u]);
              pa[u] = ld_v4(master + e[u], drop);
              pb[u] = ld_v4(master + e[u] + 4, drop);
            }
          }
        }
#pragma unroll
        for (int u = 0; u < kU2; ++u) {
          const int i = i0 + u * kThreads;
          if (full[u]) {
            uint4 o0, o1, ob;
            uint2 ocm, ocv;
            phase2_group<GT>(c, r[u], pa[u], pb[u], o0, o1, ob, ocm, ocv);
            st_v4(master + e[u], o0, drop);
            st_v4(master + e[u] + 4, o1, drop);
            st_v4(bf + e[u], ob, drop);
            st_v2(mq + e[u], ocm, drop);
            st_v2(vq + e[u], ocv, drop);
          } else if (i < sh.ngroups) {
            phase2_scalar<GT>(c, grad, mq, vq, master, bf, e[u], cnt[u]);
          }
        }
      }
    } else {
      for (int rr = warp; rr < sh.ngroups; rr += kWarps) {
        const int64_t row = sh.base + (sh.first + rr) * (int64_t)sh.stride;
        for (int v = lane; v < vpr; v += 32)
          phase2_scalar<GT>(c, grad, mq, vq, master, bf, row + v * 8, min(8, sh.ncols - v * 8));
      }
    }
  }
  __syncwarp();
  cluster.sync();  // no CTA leaves while a peer may still write its slots
}

// Element-granular chunks (g_coll elements each): one warp per block, two
// passes over the (cache-resident) chunk.
template <typename GT>
__global__ void __launch_bounds__(kSmallThreads) adam_small_kernel(
    const QBlock* __restrict__ qb, const int32_t* __restrict__ list, int nlist,
    const GT* __restrict__ grad, const float* __restrict__ d_factor, float* master, int8_t* mq,
    uint8_t* vq, float* m_scale, float* v_scale, uint16_t* bf, AdamConsts k) {
  // The bulk-copy kernel, launched next with programmatic serialization,
  // touches other blocks only: let it start at once.
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  const int lane = threadIdx.x & 31;
  const int j = blockIdx.x * (kSmallThreads / 32) + (threadIdx.x >> 5);
  if (j >= nlist) return;
  const int q = list[j];
  const QBlock b = qb[q];
  if (!in_bounds(k.bd, b.base, b.base + b.ncols)) return;
  Consts2 c;
  c.b1 = f2(k.b1);
  c.omb1 = f2(k.omb1);
  c.b2 = f2(k.b2);
  c.omb2 = f2(k.omb2);
  c.eps_hat = f2(k.eps_hat);
  c.decay = f2(k.decay);
  c.alpha = f2(k.alpha);
  c.factor = f2(*d_factor);
  c.dm = f2(__fdiv_rn(m_scale[q], 127.0f));
  c.dv = f2(__fdiv_rn(v_scale[q], 255.0f));
  float mx = 0.0f, vx = 0.0f;
  for (int i = lane; i < b.ncols; i += 32) phase1_scalar<GT>(c, grad, mq, vq, b.base + i, 1, mx, vx);
  const float sm = warp_max(mx), sv = warp_max(vx);
  c.im = f2(sm > 0.0f ? __fdiv_rn(127.0f, sm) : 0.0f);
  c.iv = f2(sv > 0.0f ? __fdiv_rn(255.0f, sv) : 0.0f);
  for (int i = lane; i < b.ncols; i += 32)
    phase2_scalar<GT>(c, grad, mq, vq, master, bf, b.base + i, 1);
  __syncwarp();
  if (lane == 0) {
    m_scale[q] = sm;
    v_scale[q] = sv;
  }
}

// fp32 moments (no quantisation): element-wise over the copy spans.
template <typename GT>
__global__ void __launch_bounds__(kCopyThreads) adam_fp32_kernel(
    const int64_t* __restrict__ t_off, const int64_t* __restrict__ t_lo, const int64_t* __restrict__ t_hi,
    const CopySpan* __restrict__ spans, const GT* __restrict__ grad,
    const float* __restrict__ d_factor, float* master, float* m_state, float* v_state,
    uint16_t* bf, AdamConsts k) {
  const CopySpan s0 = spans[blockIdx.x];
  const CopySpan s1 = spans[blockIdx.x + 1];
  Consts2 c;
  c.b1 = f2(k.b1);
  c.omb1 = f2(k.omb1);
  c.b2 = f2(k.b2);
  c.omb2 = f2(k.omb2);
  c.eps_hat = f2(k.eps_hat);
  c.decay = f2(k.decay);
  c.alpha = f2(k.alpha);
  c.factor = f2(*d_factor);
  c.dm = f2(1.0f);
  c.dv = f2(1.0f);
  for (int t = s0.tensor; t <= s1.tensor; ++t) {
    const int64_t b = (t == s0.tensor) ? s0.elem : t_lo[t];
    const int64_t e = (t == s1.tensor) ? s1.elem : t_hi[t];
    const int64_t base = t_off[t];
    if (b < e && !in_bounds(k.bd, base + b, base + e)) continue;
    for (int64_t i = b + threadIdx.x; i < e; i += kCopyThreads) {
      const int64_t x = base + i;
      float m, v;
      // with dm = dv = 1 the "dequantised" moments are the fp32 state itself
      moments1(c, elem_f32(grad[x]), m_state[x], v_state[x], m, v);
      const float p = update1(c, master[x], m, v);
      m_state[x] = m;
      v_state[x] = v;
      master[x] = p;
      bf[x] = (uint16_t)bf16_bits(p);
    }
  }
}
