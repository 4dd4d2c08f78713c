/*
 * vsf.h — C ABI of libvsf: the local per-step data path of structure-aware
 * FSDP on one GB300 (sm_103a), with all m virtual ranks in one buffer.
 *
 * Sources, cited by page title and section:
 *   [VSF]  "veScale-FSDP: Flexible and High-Performance FSDP at Scale
 *          (MLSys 2026)" summary page:
 *            核心方法 › RaggedShard            (atoms: element / row / 2-D block)
 *            核心方法 › Grouped communication  (Algorithm 1: layout planning)
 *            核心方法 › Distributed Buffer     (one global buffer, fused group
 *                                               ops add/scale/zero/copy, fixed
 *                                               address map)
 *            结构感知训练 case study › 8-bit Adam (per-block quantisation kept
 *                                               local by intact blocks)
 *   [FSDP] "FSDP" concept page › 关键观察 (copy-in / copy-out cost around the
 *          collective buffer).
 *
 * Conventions for every call:
 *   - Every function returns a vsf_status; no exception crosses the ABI.
 *     vsf_last_error() gives a thread-local message for the last failure.
 *   - The plan and its host tables are owned by the library. ALL device
 *     memory (workspace, buffers, per-tensor tensors) is owned by the caller;
 *     the library never allocates device memory and never synchronises.
 *   - Device pointers must be 16-byte aligned (VSF_ERR_ALIGN otherwise).
 *   - `stream` is a cudaStream_t passed as void* (NULL = legacy default
 *     stream). Kernels are enqueued asynchronously on it; a launch failure is
 *     VSF_ERR_CUDA.
 *   - Buffers indexed by "buffer element" hold m*S elements (see
 *     vsf_plan_info.total); virtual rank r owns elements [r*S, (r+1)*S).
 *     A plan restricted to ranks [r0, r1) (vsf_plan_restrict) uses buffers
 *     of (r1 - r0)*S elements holding [r0*S, r1*S). Padding elements are
 *     never read or written by the per-step calls.
 */
#ifndef VSF_H
#define VSF_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef int32_t vsf_status;
enum {
  VSF_OK = 0,
  VSF_ERR_ARG = -1,        /* bad argument or descriptor */
  VSF_ERR_INFEASIBLE = -2, /* no layout found */
  VSF_ERR_OVERFLOW = -3,   /* sizes overflow 64-bit element indices */
  VSF_ERR_ALIGN = -4,      /* a device pointer is not 16-byte aligned */
  VSF_ERR_CUDA = -5,       /* a CUDA call or kernel launch failed */
  VSF_ERR_STATE = -6       /* call out of order (e.g. plan not uploaded) */
};

/* Shard atom of a tensor ([VSF] 核心方法 › RaggedShard). A tensor of shape
 * [d0 .. dk-1] is viewed as R = d0*..*dk-2 rows of C = dk-1 elements.
 *   ELEM: atom = 1 element; quantisation blocks are g_coll consecutive
 *         elements from the tensor start.
 *   ROWS: atom = block_rows whole rows; one quantisation block per atom.
 *   TILE: atom = block_rows whole rows (a stripe); one quantisation block
 *         per block_rows x tile_cols tile of the stripe.
 * The last block of a tensor may be short. */
enum { VSF_GRAN_ELEM = 0, VSF_GRAN_ROWS = 1, VSF_GRAN_TILE = 2 };

/* Tensor order tried by the planner ([VSF] Algorithm 1, first step): input
 * order, atom size descending, element count descending (ties keep input
 * order), or the best of the three (ties prefer the earlier one). */
enum { VSF_ORDER_DEFAULT = 0, VSF_ORDER_BLOCK = 1, VSF_ORDER_SHAPE = 2, VSF_ORDER_BEST3 = 3 };

/* Element type of gradients (per-tensor and packed). Parameters are bf16. */
enum { VSF_BF16 = 0, VSF_FP32 = 1 };

typedef struct {
  int32_t ndim;       /* 1..8 */
  int32_t gran;       /* VSF_GRAN_* */
  int64_t shape[8];   /* shape[0..ndim) */
  int64_t block_rows; /* ROWS / TILE: rows per atom; ignored for ELEM */
  int64_t tile_cols;  /* TILE: columns per quantisation tile */
} vsf_tensor_desc;

/* AdamW hyper-parameters ([VSF] case study › 8-bit Adam, with the readings
 * documented for vsf_adam8_step). world = number of ranks whose gradients the
 * packed buffer sums; max_norm <= 0 or non-finite disables clipping;
 * quantized = 1 for 8-bit moments, 0 for fp32 moments. */
typedef struct {
  double lr, beta1, beta2, eps, weight_decay, max_norm;
  int32_t world;
  int32_t quantized;
} vsf_adam_hparams;

typedef struct {
  int64_t S;             /* uniform per-rank size in elements */
  int64_t total;         /* elements of every packed buffer: (rank_end - rank_begin) * S */
  int64_t real;          /* real (non-padding) elements inside the rank window */
  int64_t n_qblocks;     /* quantisation blocks in the window = entries of m_scale / v_scale */
  int32_t n_tensors, m;
  int64_t g_coll;
  double padding_ratio;  /* 1 - real / total */
  double plan_seconds;   /* host time spent in vsf_plan_create */
  int32_t order_used;    /* VSF_ORDER_* actually chosen */
  int32_t bulk_warps;    /* consumer warps per CTA of the bulk-copy AdamW kernel:
                          * 16 (one CTA per SM), or 4 (four CTAs per SM) when
                          * every bulk-copy unit has at most 49152 elements */
  /* how vsf_adam8_step splits the blocks (each non-zero count is one launch):
   * bulk-copy work units (contiguous blocks, or k full tiles), blocks of the
   * register kernel (ragged or unaligned), element-granular chunks */
  int64_t n_bulk_units, n_register_blocks, n_element_chunks;
  int32_t rank_begin, rank_end; /* the plan's rank window (0, m unless restricted) */
  int32_t bulk_cluster;  /* CTAs per thread-block cluster of the bulk-copy AdamW
                          * kernel (1, 2, 4 or 8), chosen by vsf_plan_upload
                          * from the units' sizes and the GPU; 0 before upload */
  int32_t reserved;      /* 0 */
} vsf_plan_info;

typedef struct vsf_plan vsf_plan; /* opaque */

/* Plans the layout ([VSF] 核心方法 › Grouped communication, Algorithm 1): the
 * smallest uniform per-rank size S, a multiple of g_coll and at least
 * ceil(real/m), such that tensors placed one after another in the chosen
 * order, each at the earliest offset that is a multiple of lcm(g_coll, atom)
 * and that no rank boundary k*S cuts inside an atom, end within m*S. Padding
 * sits only between tensors. Host only; no CUDA call.
 * Errors: VSF_ERR_ARG (bad descriptor, n < 1, m < 1, g_coll < 1),
 * VSF_ERR_OVERFLOW, VSF_ERR_INFEASIBLE. On success *out owns a new plan. */
vsf_status vsf_plan_create(const vsf_tensor_desc* descs, int32_t n, int32_t m, int64_t g_coll,
                           int32_t order, vsf_plan** out);
void vsf_plan_destroy(vsf_plan* plan);

/* Restricts a plan, before vsf_plan_upload, to the virtual ranks
 * [rank_begin, rank_end): the part of the DBuffer one process owns ([VSF]
 * 核心方法 › RaggedShard and Distributed Buffer: each rank holds its own
 * slice; no quantisation block crosses a rank boundary, so every block lies
 * in one window). The layout (S, offsets) is unchanged. Afterwards:
 *   - every packed buffer passed to a per-step call holds the window, i.e.
 *     elements [rank_begin*S, rank_end*S) of the planned buffer, indexed from
 *     0 (total = (rank_end - rank_begin) * S);
 *   - vsf_pack / vsf_unpack / group ops touch only the window's elements
 *     (per-tensor tensors stay whole: element i of tensor t is copied when
 *     offset_t + i falls in the window);
 *   - the quantisation-block table, n_qblocks and the scale arrays cover the
 *     window's blocks only, with bases counted from the window start;
 *   - the gradient norm needs every window: vsf_group_sumsq gives this
 *     window's sum of squares, the caller adds the windows' sums (an
 *     all-reduce of one fp64 value), and vsf_group_scale_from_sumsq turns the
 *     total into the factor. vsf_group_norm_scale, vsf_plan_views and
 *     vsf_muon_step need whole tensors and return VSF_ERR_STATE.
 * Calling it again replaces the window. Errors: VSF_ERR_ARG (NULL plan, not
 * 0 <= rank_begin < rank_end <= m), VSF_ERR_STATE (already uploaded). */
vsf_status vsf_plan_restrict(vsf_plan* plan, int32_t rank_begin, int32_t rank_end);

/* Shape of the bulk-copy AdamW kernel (vsf_plan_info.bulk_warps). warps = 16
 * (wide: one CTA per SM) or 4 (narrow: four CTAs per SM) forces that shape;
 * 0 restores the planner's choice (narrow when every bulk-copy unit has at
 * most 49152 elements and the narrow copy boxes keep every unit). Results are
 * identical in either shape; only speed differs. A forced narrow shape may
 * send tile units whose stripe height its 8-row copy box does not divide to
 * the register kernel. Rebuilds the tables for the plan's rank window and
 * stays in force across vsf_plan_restrict. Host only.
 * Errors: VSF_ERR_ARG (NULL plan, warps not 0, 4 or 16), VSF_ERR_STATE
 * (already uploaded). */
vsf_status vsf_plan_set_bulk_warps(vsf_plan* plan, int32_t warps);

vsf_status vsf_plan_get_info(const vsf_plan* plan, vsf_plan_info* info);

/* Checkpointing a plan. The layout is a deterministic function of the
 * descriptors, m, g_coll and the order policy ([VSF] 核心方法 › Grouped
 * communication, Algorithm 1), so a plan is stored as those inputs plus
 * its rank window and forced kernel shape, and the S and offsets it
 * produced (to check against on load). Host only; no CUDA call.
 *
 * vsf_plan_serialize writes the plan into buf. With buf == NULL it only sets
 * *bytes to the size needed. Otherwise *bytes is the capacity of buf on
 * entry and the size written on return. Errors: VSF_ERR_ARG (NULL plan or
 * bytes; capacity too small, *bytes then set to the size needed). The
 * format is the host's native byte order (little-endian on x86-64 and
 * Arm64), versioned, with a 64-bit FNV-1a checksum.
 *
 * vsf_plan_deserialize plans again from the stored inputs, checks that S and
 * every offset equal the stored ones, restricts to the stored rank window and
 * forces the stored kernel shape. The result is a new, not yet uploaded plan
 * in *out. Errors: VSF_ERR_ARG (NULL, truncated buffer, bad magic, version
 * or checksum, inconsistent sizes), VSF_ERR_STATE (the planner now gives
 * another layout for the same inputs), and the errors of vsf_plan_create. */
vsf_status vsf_plan_serialize(const vsf_plan* plan, void* buf, size_t* bytes);
vsf_status vsf_plan_deserialize(const void* buf, size_t bytes, vsf_plan** out);

/* Per-tensor element offsets into the m*S buffer; offsets has n entries. */
vsf_status vsf_plan_offsets(const vsf_plan* plan, int64_t* offsets);

/* Quantisation-block table, in tensor order then stripe, then tile: block q
 * is the row-major region of nrows rows x ncols elements starting at buffer
 * element base[q] (counted from the rank window's start), rows `stride`
 * elements apart, of tensor tensor[q]. Arrays have n_qblocks entries (any
 * may be NULL). */
vsf_status vsf_plan_qblocks(const vsf_plan* plan, int32_t* tensor, int64_t* base, int64_t* nrows,
                            int64_t* ncols, int64_t* stride);

/* RaggedShard slice of virtual rank `rank` ([VSF] 核心方法 › RaggedShard:
 * uneven, whole atoms): for each tensor overlapping [rank*S, (rank+1)*S), in
 * buffer order, the tensor index, its element range [elem_begin, elem_end)
 * and its atom range [atom_begin, atom_end). Writes at most `capacity`
 * entries and the full count into *count (call with capacity 0 to size). */
vsf_status vsf_plan_rank_slices(const vsf_plan* plan, int32_t rank, int32_t capacity,
                                int32_t* count, int32_t* tensor, int64_t* elem_begin,
                                int64_t* elem_end, int64_t* atom_begin, int64_t* atom_end);

/* The persistent address map ([VSF] 核心方法 › Distributed Buffer: zero-copy
 * access to every parameter's data around the collectives): views[t] =
 * packed + offset_t * elem_bytes, for a packed buffer of 1-, 2- or 4-byte
 * elements. A caller that lets its per-tensor gradients and parameters BE
 * these views (zero-copy mode) skips vsf_pack and vsf_unpack: one step is
 * then vsf_group_norm_scale on the packed gradient and vsf_adam8_step. Host
 * pointer arithmetic only. */
vsf_status vsf_plan_views(const vsf_plan* plan, const void* packed, int32_t elem_bytes,
                          void** views);

/* Bytes of device workspace the caller must provide to vsf_plan_upload. */
size_t vsf_plan_workspace_bytes(const vsf_plan* plan);

/* Byte offset, inside the workspace, of a 32-bit device error word (zeroed
 * by vsf_plan_upload). A kernel sets bit 1 when one of its bounded waits
 * runs out (the step's results are then not to be trusted); the caller reads
 * it with an ordinary device-to-host copy after synchronising the stream. */
vsf_status vsf_plan_device_error_offset(const vsf_plan* plan, size_t* offset);

/* Copies the plan's device tables into the caller's workspace (16-byte
 * aligned, vsf_plan_workspace_bytes long) on `stream`, zeroes its scratch,
 * and binds the plan to the current CUDA device. Must precede every per-step
 * call; the workspace must stay allocated while the plan is used. Calls that
 * share one plan (and so one workspace) must be ordered on the device. The
 * first upload on a device also creates the plan's own non-blocking streams
 * (three) and events, which vsf_muon_step forks onto; vsf_plan_destroy
 * releases them. */
vsf_status vsf_plan_upload(vsf_plan* plan, void* d_workspace, size_t bytes, void* stream);

/* Copy-in with the fused squared-norm reduction ([FSDP] 关键观察; [VSF]
 * Distributed Buffer, group copy): packed_grad[offset_t + i] = grads[t][i]
 * for every real element. grads is a HOST array of n device pointers, each
 * 16-byte aligned, of the tensor's element type (dtype VSF_BF16 or
 * VSF_FP32); packed_grad has m*S elements of that type. Also leaves per-CTA
 * fp64 partial sums of g^2 in the workspace for vsf_group_norm_scale. */
vsf_status vsf_pack(const vsf_plan* plan, const void* const* grads, int32_t dtype,
                    void* packed_grad, void* stream);

/* Group norm and scale ([VSF] Distributed Buffer, fused group scale):
 * sumsq = sum of g^2 over every real element (fp64); norm = sqrt(sumsq) /
 * world (the norm of the mean gradient, the packed buffer being the sum over
 * `world` ranks); c = min(1, max_norm / (norm + 1e-6)) when clipping is on,
 * else 1; writes *d_factor = fp32(c / world) and *d_norm = norm (both device
 * pointers; d_norm may be NULL). With packed_grad == NULL the partial sums
 * left by the last vsf_pack on this plan are used; otherwise they are
 * recomputed from packed_grad (element type dtype). A plan restricted to a
 * rank window gets VSF_ERR_STATE: its norm needs the other windows. */
vsf_status vsf_group_norm_scale(const vsf_plan* plan, const void* packed_grad, int32_t dtype,
                                const vsf_adam_hparams* hp, float* d_factor, double* d_norm,
                                void* stream);

/* The same norm split at its one cross-rank exchange, for plans restricted
 * to a rank window (vsf_plan_restrict). vsf_group_sumsq writes the window's
 * fp64 sum of g^2 to *d_sumsq (device), from the last vsf_pack's partials
 * (packed_grad == NULL) or from packed_grad. vsf_group_scale_from_sumsq takes
 * the total over all windows (device fp64; the caller's all-reduce) and
 * writes *d_factor and *d_norm exactly as vsf_group_norm_scale does; it needs
 * no plan. Errors: VSF_ERR_ARG (NULL, world < 1, bad dtype), VSF_ERR_ALIGN,
 * VSF_ERR_STATE (plan not uploaded), VSF_ERR_CUDA. */
vsf_status vsf_group_sumsq(const vsf_plan* plan, const void* packed_grad, int32_t dtype,
                           double* d_sumsq, void* stream);
vsf_status vsf_group_scale_from_sumsq(const double* d_sumsq, const vsf_adam_hparams* hp,
                                      float* d_factor, double* d_norm, void* stream);

/* Block-wise 8-bit AdamW on every virtual rank's RaggedShard slice ([VSF]
 * case study › 8-bit Adam; blocks never cross a rank, so every scale is
 * local). Per element, in fp32 with every operation rounded once:
 *   g = factor * grad;  m = b1*m' + (1-b1)*g;  v = b2*v' + (1-b2)*g*g;
 *   p = p * (1 - lr*wd);  p = p - step_size * (m / (sqrt(v)/bc2s + eps)),
 *   step_size = lr / (1 - b1^step), bc2s = sqrt(1 - b2^step), the constants
 *   computed in double and rounded once to fp32; bf16 = RNE(p).
 * quantized = 1: m' = code_m * (m_scale[q] / 127), v' = code_v *
 *   (v_scale[q] / 255); after the update each block q gets m_scale[q] =
 *   max|m|, v_scale[q] = max v and codes round-half-even(m * (127/m_scale)),
 *   clamped to [-127, 127] (int8), and round-half-even(v * (255/v_scale)),
 *   clamped to [0, 255] (uint8); a zero scale gives all-zero codes.
 *   m_state / v_state: int8 / uint8 arrays of m*S; m_scale / v_scale: fp32
 *   arrays of n_qblocks. Initial state: codes 0, scales 0, step 1.
 * quantized = 0: m_state / v_state are fp32 arrays of m*S; scales unused.
 * packed_grad: m*S elements of grad_dtype; d_factor: device fp32 scalar (from
 * vsf_group_norm_scale); master: fp32 m*S (in/out); packed_bf16: bf16 bits,
 * m*S (out). step >= 1.
 * Errors: VSF_ERR_ARG (NULL pointer, step < 1, bad grad_dtype),
 * VSF_ERR_ALIGN, VSF_ERR_STATE (plan not uploaded), VSF_ERR_CUDA (tensor-map
 * encoding or a launch). Every error but a failed launch is found before the
 * first launch, so the buffers are untouched. A failed launch may follow a
 * successful one, so the state buffers of that step are then undefined.
 * Kernel-side failures (a bounded wait that timed out, a failed index check
 * in the bounds-checking build) set bits in the plan's device error word
 * (vsf_plan_device_error_offset). */
vsf_status vsf_adam8_step(const vsf_plan* plan, const void* packed_grad, int32_t grad_dtype,
                          const float* d_factor, float* master, void* m_state, void* v_state,
                          float* m_scale, float* v_scale, uint16_t* packed_bf16,
                          const vsf_adam_hparams* hp, int32_t step, void* stream);

/* Copy-out ([FSDP] 关键观察; [VSF] Distributed Buffer, group copy):
 * params[t][i] = packed_bf16[offset_t + i]. params is a HOST array of n
 * device pointers (bf16, 16-byte aligned). */
vsf_status vsf_unpack(const vsf_plan* plan, const uint16_t* packed_bf16, void* const* params,
                      void* stream);

/* Measurement helper: a plain device-to-device copy of `bytes` bytes by a
 * streaming kernel (128-bit loads and stores, a grid of 4 CTAs of 512
 * threads per SM, 8 accesses in flight per thread). It sets the copy ceiling
 * that the shard-step kernels are measured against in the same run. dst and
 * src are device pointers, 16-byte aligned, not overlapping; bytes a
 * multiple of 16. Errors: VSF_ERR_ARG (NULL, bytes not a multiple of 16),
 * VSF_ERR_ALIGN, VSF_ERR_CUDA. */
vsf_status vsf_device_copy(void* dst, const void* src, size_t bytes, void* stream);

/* Fused group ops ([VSF] 核心方法 › Distributed Buffer: the same
 * element-wise kernel applied to every tensor of the buffer in one launch,
 * e.g. zero_grad and gradient accumulation). They touch every real element
 * of the m*S packed buffer(s) and never the padding. Arithmetic in fp32 with
 * one rounding, then the destination type (bf16: round half to even).
 *   vsf_group_zero:  buf = 0
 *   vsf_group_scale: buf = buf * alpha
 *   vsf_group_add:   dst = dst + src (gradient accumulation; any mix of
 *                    VSF_BF16 / VSF_FP32 destination and source)
 * Buffers are device pointers, 16-byte aligned, of m*S elements. */
vsf_status vsf_group_zero(const vsf_plan* plan, void* buf, int32_t dtype, void* stream);
vsf_status vsf_group_scale(const vsf_plan* plan, void* buf, int32_t dtype, float alpha,
                           void* stream);
vsf_status vsf_group_add(const vsf_plan* plan, void* dst, int32_t dst_dtype, const void* src,
                         int32_t src_dtype, void* stream);

/* Distributed Muon ([VSF] 结构感知训练 case study › 分布式 Muon, Algorithm 2)
 * on every matrix tensor of the plan (ndim >= 2; leading dims index a batch
 * of matrices); 1-D tensors are left untouched.
 *   SelectRoot: vsf_muon_select_roots gives each matrix tensor a root virtual
 *   rank (longest-processing-time greedy over the Newton-Schulz FLOPs; -1 for
 *   1-D tensors) and the max/mean root load.
 *   Redistribute to the root and back is zero-copy here: a tensor is
 *   contiguous in the buffer.
 *   vsf_muon_step, per matrix, all in fp32 rounded once per operation except
 *   the tensor-core products (bf16 operands, fp32 accumulation, bf16 results):
 *     M = mu M + g;  U = g + mu M (Nesterov);
 *     X = bf16(U * fp32(1 / (||U||_F + eps)));
 *     ns_steps times: A = X X^T (R <= C) or X^T X (R > C); B = c A A + b A;
 *                     X = a X + B X (R <= C) or a X + X B (R > C);
 *     p = p (1 - lr wd) - fp32(lr sqrt(max(1, R/C))) X;  bf16 copy.
 *   packed_grad: bf16, m*S; momentum: fp32, m*S (caller-zeroed before step
 *   1); master: fp32; packed_bf16: out. d_workspace: vsf_muon_workspace_bytes
 *   of caller memory (per stream lane, the Newton-Schulz operands X, X', A, B
 *   of its largest batch and the norm partials). The products run on the
 *   library's tcgen05 kernel (vsf_ns_gemm below); its bounded waits report
 *   through the plan's device error word. Matrices of one shape, across
 *   tensors, run batched: vsf_muon_chunk_count gives the number of batches
 *   (each: 3 element-wise kernels and 3 * ns_steps products); 0 for a NULL
 *   plan. The batches are independent and run on four stream lanes:
 *   `stream` itself and the plan's own three streams, which wait for
 *   `stream`'s earlier work (an event) and which `stream` waits for before
 *   its later work, so the call is ordered on `stream` like a single launch
 *   (also under stream capture). Errors:
 *   VSF_ERR_ARG (NULL, small workspace, ns_steps < 0), VSF_ERR_ALIGN (a
 *   pointer not 16-byte aligned), VSF_ERR_STATE (plan not uploaded),
 *   VSF_ERR_CUDA (a launch or a tensor-map encoding failed).
 *   Argument errors are found before the first launch (buffers untouched);
 *   after VSF_ERR_CUDA, chunks before the failing one have been updated and
 *   the step's momentum, master and bf16 buffers are undefined. */
typedef struct {
  double lr, momentum, weight_decay, eps, ns_a, ns_b, ns_c;
  int32_t ns_steps, reserved;
} vsf_muon_hparams;

vsf_status vsf_muon_select_roots(const vsf_plan* plan, int32_t* root, double* load_balance);
size_t vsf_muon_workspace_bytes(const vsf_plan* plan);
int32_t vsf_muon_chunk_count(const vsf_plan* plan);
/* Launches of the library's own kernels in one vsf_muon_step with ns_steps
 * iterations: per batched chunk, momentum, normalisation and update, plus the
 * three Newton–Schulz products of every iteration. 0 for a NULL plan. */
int64_t vsf_muon_kernel_launches(const vsf_plan* plan, int32_t ns_steps);
vsf_status vsf_muon_step(const vsf_plan* plan, const uint16_t* packed_grad, float* momentum,
                         float* master, uint16_t* packed_bf16, const vsf_muon_hparams* hp,
                         void* d_workspace, size_t ws_bytes, void* stream);

/* One Newton–Schulz product of distributed Muon ([VSF] 结构感知训练 case study
 * › 分布式 Muon, Algorithm 2: the root's orthogonalisation needs A = X X^T (or
 * X^T X), B = c A A + b A and X' = a X + B X (or a X + X B)), as the
 * library's tcgen05 tensor-core kernel computes it inside vsf_muon_step:
 *   D[b] = alpha * opA[b] * opB[b]^T + beta * C[b],  b = 0 .. batch-1,
 * opA M x K, opB N x K, C and D M x N. All matrices are bf16, row-major, with
 * leading dimension ld* and batch stride s* in elements; accumulation is fp32
 * and D is rounded to nearest even once, after alpha * acc + beta * C.
 *   a_mn = 0: opA[i][k] = A[i*lda + k] (K-major); a_mn = 1: A[k*lda + i]
 *   (MN-major); likewise b_mn for opB[j][k]. Supported: K/K, K/MN, and MN/MN
 *   with sym = 1.
 *   sym = 1 (requires M = N and opA = opB, with C symmetric when beta != 0):
 *   only the output tiles that reach or lie above the diagonal are computed
 *   (half of the FLOPs); every D[i][j] with i <= j is written to D[i][j] and
 *   D[j][i], so D is exactly symmetric.
 *   C is read only when beta != 0 (may be NULL otherwise); D must not overlap
 *   A, B or C. d_err: the device error word that a bounded wait sets (bit 1)
 *   if the kernel's pipeline ever stalls for 2 s; a correct launch leaves it
 *   unchanged.
 * The tensor-core kernel needs 16-byte aligned A, B, C, D and leading
 * dimensions and batch strides that are multiples of 8; other operands run a
 * plain CUDA-core kernel with the same contract. Asynchronous on `stream`.
 * Errors: VSF_ERR_ARG (NULL, sizes out of range, unsupported layout),
 * VSF_ERR_CUDA. */
vsf_status vsf_ns_gemm(int32_t a_mn, int32_t b_mn, int32_t sym, int64_t M, int64_t N, int64_t K,
                       int64_t batch, const uint16_t* A, int64_t lda, int64_t sa, const uint16_t* B,
                       int64_t ldb, int64_t sb, float alpha, float beta, const uint16_t* C,
                       int64_t ldc, int64_t sc, uint16_t* D, int64_t ldd, int64_t sd,
                       unsigned* d_err, void* stream);

/* Self-test of the kernels' bounded waits (every wait on a barrier gives up
 * after a time limit, sets bit 1 of the device error word and lets the kernel
 * finish, so no thread can hang; the first timeout in a CTA makes every later
 * wait of that CTA return at once): launches one CTA that waits four times
 * in a row on barriers nobody arrives on, with limit_ns (at most 1 s) instead
 * of the kernels' 2 s. d_err points to two device uint32 words the caller
 * zeroed. After the stream reaches the kernel, d_err[0] has bit 1 set and
 * d_err[1] holds the four waits' elapsed time in microseconds: about one
 * limit, as the timeout is sticky. Errors: VSF_ERR_ARG (NULL, limit above
 * 1 s), VSF_ERR_CUDA. */
vsf_status vsf_selftest_wait_timeout(unsigned* d_err, uint64_t limit_ns, void* stream);

/* Group norm and scale WITHOUT any device allocation or workspace. The pages
 * have no counterpart: this entry point exists for callers that cannot
 * allocate device memory where they need the gradient norm, such as a hook
 * running inside a framework's caching allocator (its out-of-memory or
 * reclaim path, where asking for memory would recurse into the allocator), a
 * runtime that owns the whole device memory budget and forbids raw
 * cudaMalloc, or latency-critical code that cannot pay for the device
 * synchronisation cudaMalloc / cudaFree may imply.
 *   grads: HOST array of n device pointers (16-byte aligned) to the gradient
 *   tensors, element type dtype (VSF_BF16 or VSF_FP32); numel: HOST array of
 *   their element counts (each >= 1); 1 <= n <= 1024 (VSF_ERR_ARG beyond).
 *   Computes what vsf_group_norm_scale computes (sum of g^2 over every
 *   element, norm = sqrt(sum) / world, clip factor, *d_factor = fp32(c /
 *   world), *d_norm = norm; d_norm may be NULL) on `stream`.
 * Scratch: a fixed 8 KB array of per-CTA partial sums (at most 1024 CTAs)
 * that the library declares at file scope in device memory; every device
 * that loads the library keeps it until the process exits. No cudaMalloc,
 * cudaFree or allocating library call is made. The first call on a device
 * looks up the array's device address for that device (with that device
 * current) and caches it with the current context; make that first call
 * before any stream capture. After a device reset (a new primary context),
 * the next call looks the address up again, so it too belongs outside a
 * capture.
 * Every call on a device shares the array: calls that overlap on the GPU
 * (different streams without ordering) race and give wrong results. Nothing
 * needs to start at zero: each call writes every partial it later reads. */
vsf_status vsf_group_norm_scale_static(const void* const* grads, const int64_t* numel, int32_t n,
                                       int32_t dtype, const vsf_adam_hparams* hp, float* d_factor,
                                       double* d_norm, void* stream);

const char* vsf_status_string(vsf_status s);
const char* vsf_last_error(void);

#ifdef __cplusplus
}
#endif

#endif /* VSF_H */
