"""ShardStep: device buffers of one planned DBuffer (allocated with torch)
and the four per-step calls of libvsf, in order, on one CUDA stream.

Argument marshalling only: every step of the path runs in libvsf's kernels.
"""
from __future__ import annotations

import dataclasses

import torch

from . import vsf as V


@dataclasses.dataclass
class TensorSpec:
    shape: tuple
    gran: int
    block_rows: int = 0
    tile_cols: int = 0


class ShardStep:
    """One DBuffer of m virtual ranks on the current CUDA device.

    With ranks=(r0, r1) the plan is restricted to virtual ranks [r0, r1): the
    packed buffers hold that window only ((r1 - r0) * S elements) and the
    norm is split (group_sumsq, an all-reduce by the caller, scale_from_sumsq).

    Buffers (m*S elements each unless noted): packed_grad (bf16 or fp32),
    master (fp32), m_state / v_state (int8 / uint8 codes, or fp32 when
    quantized=False), m_scale / v_scale (fp32, one per quantisation block),
    packed_bf16 (bf16 bits), factor (fp32 scalar), norm (fp64 scalar).
    """

    def __init__(self, specs, m: int, g_coll: int, *, order: int = V.VSF_ORDER_DEFAULT,
                 grad_dtype: int = V.VSF_BF16, quantized: bool = True, lr=1e-3, beta1=0.9,
                 beta2=0.999, eps=1e-8, weight_decay=0.01, max_norm=float("inf"),
                 world: int | None = None, device=None, stream: torch.cuda.Stream | None = None,
                 ranks: tuple[int, int] | None = None, bulk_warps: int = 0):
        self.specs = list(specs)
        self.m, self.g_coll = m, g_coll
        self.grad_dtype = grad_dtype
        self.quantized = quantized
        descs = [V.make_desc(s.shape, s.gran, s.block_rows, s.tile_cols) for s in self.specs]
        self.plan = V.vsf_plan_create(descs, m, g_coll, order)
        if ranks is not None:  # this process owns virtual ranks [r0, r1) only
            V.vsf_plan_restrict(self.plan, int(ranks[0]), int(ranks[1]))
        if bulk_warps:  # force a bulk-copy AdamW kernel shape (4 or 16); results are the same
            V.vsf_plan_set_bulk_warps(self.plan, int(bulk_warps))
        self.info = V.vsf_plan_get_info(self.plan)
        self.offsets = V.vsf_plan_offsets(self.plan, len(self.specs))
        self.numels = [int(torch.Size(s.shape).numel()) for s in self.specs]
        self.hp = V.make_hparams(lr, beta1, beta2, eps, weight_decay, max_norm,
                                 m if world is None else world, int(quantized))
        self.device = torch.device("cuda", torch.cuda.current_device()) if device is None \
            else torch.device(device)
        self.stream = stream if stream is not None else torch.cuda.current_stream(self.device)
        total, nq = self.info.total, self.info.n_qblocks
        dev = self.device
        gdt = torch.bfloat16 if grad_dtype == V.VSF_BF16 else torch.float32
        with torch.cuda.device(dev):
            self.workspace = torch.empty(V.vsf_plan_workspace_bytes(self.plan), dtype=torch.uint8,
                                         device=dev)
            self.packed_grad = torch.zeros(total, dtype=gdt, device=dev)
            self.master = torch.zeros(total, dtype=torch.float32, device=dev)
            sdt = (torch.int8, torch.uint8) if quantized else (torch.float32, torch.float32)
            self.m_state = torch.zeros(total, dtype=sdt[0], device=dev)
            self.v_state = torch.zeros(total, dtype=sdt[1], device=dev)
            self.m_scale = torch.zeros(max(nq, 1), dtype=torch.float32, device=dev)
            self.v_scale = torch.zeros(max(nq, 1), dtype=torch.float32, device=dev)
            self.packed_bf16 = torch.zeros(total, dtype=torch.bfloat16, device=dev)
            self.factor = torch.zeros(4, dtype=torch.float32, device=dev)
            self.norm = torch.zeros(2, dtype=torch.float64, device=dev)
            self.sumsq = torch.zeros(2, dtype=torch.float64, device=dev)
            V.vsf_plan_upload(self.plan, self.workspace.data_ptr(), self.workspace.numel(),
                              self.stream.cuda_stream)
        self.info = V.vsf_plan_get_info(self.plan)  # now with the upload's choices

    def close(self):
        if self.plan:
            V.vsf_plan_destroy(self.plan)
            self.plan = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    # ---- the four per-step calls (asynchronous on self.stream)
    def pack(self, grads):
        V.vsf_pack(self.plan, [g.data_ptr() for g in grads], self.grad_dtype,
                   self.packed_grad.data_ptr(), self.stream.cuda_stream)

    def group_norm_scale(self, standalone: bool = False, norm: torch.Tensor | None = None):
        """Factor into self.factor; the fp64 norm into `norm` (a device fp64
        tensor, e.g. one slot per step of a pipeline) or else self.norm."""
        out = self.norm if norm is None else norm
        V.vsf_group_norm_scale(self.plan, self.packed_grad.data_ptr() if standalone else None,
                               self.grad_dtype, self.hp, self.factor.data_ptr(),
                               out.data_ptr(), self.stream.cuda_stream)

    def group_sumsq(self, standalone: bool = False):
        """This window's fp64 sum of squares into self.sumsq[0] (device)."""
        V.vsf_group_sumsq(self.plan, self.packed_grad.data_ptr() if standalone else None,
                          self.grad_dtype, self.sumsq.data_ptr(), self.stream.cuda_stream)

    def scale_from_sumsq(self, total: torch.Tensor):
        """Factor and norm from the sum of squares over every window (device fp64)."""
        V.vsf_group_scale_from_sumsq(total.data_ptr(), self.hp, self.factor.data_ptr(),
                                     self.norm.data_ptr(), self.stream.cuda_stream)

    def adam(self, step: int):
        V.vsf_adam8_step(self.plan, self.packed_grad.data_ptr(), self.grad_dtype,
                         self.factor.data_ptr(), self.master.data_ptr(), self.m_state.data_ptr(),
                         self.v_state.data_ptr(), self.m_scale.data_ptr(),
                         self.v_scale.data_ptr(), self.packed_bf16.data_ptr(), self.hp, step,
                         self.stream.cuda_stream)

    def unpack(self, params):
        V.vsf_unpack(self.plan, self.packed_bf16.data_ptr(), [p.data_ptr() for p in params],
                     self.stream.cuda_stream)

    def muon_step(self, hp=None):
        """Distributed Muon on every matrix tensor (packed bf16 gradient in
        self.packed_grad). Allocates the fp32 momentum buffer and the Muon
        workspace on first use."""
        if not hasattr(self, "momentum"):
            with torch.cuda.device(self.device):
                self.momentum = torch.zeros(self.info.total, dtype=torch.float32,
                                            device=self.device)
                self.muon_ws = torch.empty(V.vsf_muon_workspace_bytes(self.plan),
                                           dtype=torch.uint8, device=self.device)
        hp = V.make_muon_hparams() if hp is None else hp
        V.vsf_muon_step(self.plan, self.packed_grad.data_ptr(), self.momentum.data_ptr(),
                        self.master.data_ptr(), self.packed_bf16.data_ptr(), hp,
                        self.muon_ws.data_ptr(), self.muon_ws.numel(), self.stream.cuda_stream)

    def muon_roots(self):
        """SelectRoot: (root rank per tensor, -1 for 1-D; max/mean load)."""
        return V.vsf_muon_select_roots(self.plan, len(self.specs))

    def muon_chunks(self) -> int:
        """Batched chunks of same-shape matrices one Muon step runs."""
        return V.vsf_muon_chunk_count(self.plan)

    def adam_launches(self) -> int:
        """Kernels one vsf_adam8_step launches for this plan (quantised mode)."""
        i = self.info
        return sum(1 for c in (i.n_bulk_units, i.n_register_blocks, i.n_element_chunks) if c > 0)

    def views(self, buf: torch.Tensor):
        """Per-tensor views into a packed buffer (the persistent address map):
        writing a view writes the buffer, so pack and unpack become no-ops."""
        ptrs = V.vsf_plan_views(self.plan, buf.data_ptr(), buf.element_size(), len(self.numels))
        out = []
        for p, o, n in zip(ptrs, self.offsets, self.numels):
            v = buf[o:o + n]
            assert v.data_ptr() == p
            out.append(v)
        return out

    def zero_copy_step(self, step: int, packed_grad=None, packed_bf16=None, norm=None):
        """One step when gradients and parameters are views of the packed
        buffers: group norm/scale on the packed gradient, then AdamW. A caller
        that double-buffers passes the gradient and bf16 buffers of this step
        (same size and type as self.packed_grad / self.packed_bf16) and may
        pass a device fp64 slot for the norm; the optimizer state is always
        this object's."""
        self.zero_copy_norm(packed_grad, norm)
        self.zero_copy_adam(step, packed_grad, packed_bf16)

    def zero_copy_norm(self, packed_grad=None, norm=None):
        """The group norm/scale half of zero_copy_step (one pass over the
        packed gradient)."""
        g = self.packed_grad if packed_grad is None else packed_grad
        nrm = self.norm if norm is None else norm
        V.vsf_group_norm_scale(self.plan, g.data_ptr(), self.grad_dtype, self.hp,
                               self.factor.data_ptr(), nrm.data_ptr(),
                               self.stream.cuda_stream)

    def zero_copy_adam(self, step: int, packed_grad=None, packed_bf16=None):
        """The AdamW half of zero_copy_step."""
        g = self.packed_grad if packed_grad is None else packed_grad
        out = self.packed_bf16 if packed_bf16 is None else packed_bf16
        V.vsf_adam8_step(self.plan, g.data_ptr(), self.grad_dtype, self.factor.data_ptr(),
                         self.master.data_ptr(), self.m_state.data_ptr(), self.v_state.data_ptr(),
                         self.m_scale.data_ptr(), self.v_scale.data_ptr(), out.data_ptr(),
                         self.hp, step, self.stream.cuda_stream)

    def step(self, grads, params, step: int):
        """pack -> group norm/scale -> 8-bit AdamW -> unpack."""
        self.pack(grads)
        self.group_norm_scale()
        self.adam(step)
        self.unpack(params)

    def window_step(self, grads, params, step: int, all_reduce):
        """The step of a rank window (ranks=(r0, r1)) in one process of many:
        pack -> this window's fp64 sum of squares -> all_reduce (the sum over
        every process's window: the path's one exchange; "veScale-FSDP:
        Flexible and High-Performance FSDP at Scale (MLSys 2026)" summary
        page, 核心方法 > Distributed Buffer, fused group norm) -> factor ->
        8-bit AdamW -> unpack. all_reduce(t) sums the one-element float64
        tensor t in place across the processes (see sum_all_reduce)."""
        self.pack(grads)
        self.group_sumsq()
        total = self.sumsq[:1]
        with torch.cuda.stream(self.stream):
            all_reduce(total)
        self.scale_from_sumsq(total)
        self.adam(step)
        self.unpack(params)

    def device_error(self) -> int:
        """The device error word (0 = every bounded wait succeeded)."""
        off = V.vsf_plan_device_error_offset(self.plan)
        return int(self.workspace[off:off + 4].view(torch.int32).item())

    # ---- checkpoint / resume: the optimizer state is the caller's buffers
    STATE = ("master", "m_state", "v_state", "m_scale", "v_scale", "packed_bf16")

    def state_dict(self) -> dict:
        """Host copies of the optimizer state of this DBuffer (or rank window),
        with the plan's identity (S, offsets, rank window) to check on load."""
        torch.cuda.current_stream(self.device).wait_stream(self.stream)
        out = {k: getattr(self, k).detach().to("cpu", copy=True) for k in self.STATE}
        out["plan"] = dict(S=int(self.info.S), offsets=list(self.offsets),
                           ranks=(int(self.info.rank_begin), int(self.info.rank_end)),
                           quantized=bool(self.quantized))
        # the whole plan, from which vsf_plan_deserialize rebuilds it
        out["plan_bytes"] = V.vsf_plan_serialize(self.plan)
        return out

    def load_state_dict(self, sd: dict) -> None:
        """Restores a state_dict taken from a ShardStep with the same plan."""
        want = dict(S=int(self.info.S), offsets=list(self.offsets),
                    ranks=(int(self.info.rank_begin), int(self.info.rank_end)),
                    quantized=bool(self.quantized))
        if sd["plan"] != want:
            raise ValueError(f"state_dict was taken under another plan: {sd['plan']} != {want}")
        with torch.cuda.stream(self.stream):
            for k in self.STATE:
                getattr(self, k).copy_(sd[k], non_blocking=False)

    # ---- harness helpers
    def load_master(self, t: int, values: torch.Tensor):
        o = self.offsets[t]
        self.master[o:o + self.numels[t]].copy_(values.reshape(-1))


def sum_all_reduce(group=None):
    """all_reduce for ShardStep.window_step over a torch.distributed group:
    in place on the device with NCCL, through a host copy with gloo."""
    import torch.distributed as dist

    def reduce(t: torch.Tensor) -> None:
        if dist.get_backend(group) == "nccl":
            dist.all_reduce(t, op=dist.ReduceOp.SUM, group=group)
            return
        h = t.cpu()  # waits for the sum of squares on the current stream
        dist.all_reduce(h, op=dist.ReduceOp.SUM, group=group)
        t.copy_(h)

    return reduce
