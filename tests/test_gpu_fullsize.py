"""Parity at the full sizes of the four large workloads, in the launch
configuration the benchmark times (ShardStep: pack -> group norm/scale ->
8-bit AdamW -> unpack, every step of the workload's step count).

Checked on every workload:
  - every step: the group norm against the oracle's sum of squares over all
    real gradient elements (within the oracle's own summation error bound,
    n 2^-53 relative) and the scale factor bit for bit;
  - last step: copy-in bit for bit over every tensor (the packed gradient
    against the host gradients, padding still zero) and copy-out bit for bit
    (every parameter tensor against the packed bf16 buffer).
The optimizer state, in full on every workload: the oracle runs every
quantisation block through every step (on each tensor's real elements), and
the final master, m and v codes, m and v scales and bf16 copy of every real
element must be bit-identical (NaNs by class), and in any case within the
tolerances (master 1e-6 relative, codes |d| <= 1 at <= 1e-4 of positions).
The oracle's calls are single-threaded; each takes one run of consecutive
blocks of one tensor (blocks are independent and write disjoint elements),
and the runs go to host threads side by side, which brings the 1.3B model's
20 steps within a few minutes of host time.
"""
import os
from concurrent.futures import ThreadPoolExecutor

import numpy as np
import pytest
import torch

import oracle
from synth import workloads as W

from gpu_harness import bit_equal, check_codes, check_master

pytestmark = [pytest.mark.gpu, pytest.mark.slow]

def _tensor_blocks(qb, off_o, t):
    """The quantisation blocks of tensor t, re-based to the tensor's own
    element 0 (so that the oracle can run them on per-tensor arrays), and
    their indices in the whole plan's block table."""
    ids = np.nonzero(qb["tensor"] == t)[0]
    blocks = {k: np.ascontiguousarray(qb[k][ids]) for k in ("base", "nrows", "ncols", "stride")}
    blocks["base"] = blocks["base"] - int(off_o[t])
    return blocks, ids


def _runs(nblocks, parts):
    """[lo, hi) runs of consecutive blocks, about nblocks / parts each."""
    step = max(1, -(-nblocks // parts))
    return [(lo, min(nblocks, lo + step)) for lo in range(0, nblocks, step)]


@pytest.mark.parametrize("name", ["llama_layer", "moe_layer", "dsv3_block", "llama_1p3b"])
def test_fullsize_workload(name):
    from fsdp_buffer_layout_gb300.step import ShardStep, TensorSpec
    w = W.get(name)
    d = oracle.Desc.from_workload(w)
    S_o, off_o = oracle.plan(d, w.m, w.g_coll)
    qb = oracle.qblocks(d, w.g_coll, off_o)
    specs = [TensorSpec(t.shape, t.gran, t.block_rows, t.tile_cols) for t in w.tensors]
    ss = ShardStep(specs, w.m, w.g_coll, max_norm=w.max_norm)
    try:
        assert ss.info.S == S_o and list(ss.offsets) == [int(x) for x in off_o]
        dev = ss.device
        numels = ss.numels
        starts, cur = [], 0
        for n in numels:
            starts.append(cur)
            cur += (n + 7) // 8 * 8
        host_g = torch.zeros(cur, dtype=torch.int16).pin_memory()
        hg = host_g.numpy().view(np.uint16)
        dev_g = torch.zeros(cur, dtype=torch.int16, device=dev)
        dev_p = torch.zeros(cur, dtype=torch.int16, device=dev)
        grads = [dev_g[s:s + n] for s, n in zip(starts, numels)]
        params = [dev_p[s:s + n] for s, n in zip(starts, numels)]
        for t in range(len(specs)):
            ss.load_master(t, torch.from_numpy(W.master_init(w, t)).to(dev))

        hp = oracle.hparams(w)
        tstate = []  # the oracle's state of every tensor, tensor-local
        work = []    # (tensor, first block, end block): the oracle's calls of one step
        for t in range(d.n):
            blocks, ids = _tensor_blocks(qb, off_o, t)
            n = numels[t]
            tstate.append(dict(blocks=blocks, ids=ids, p=W.master_init(w, t).copy(),
                               mq=np.zeros(n, np.int8), vq=np.zeros(n, np.uint8),
                               msc=np.zeros(ids.size, np.float32),
                               vsc=np.zeros(ids.size, np.float32),
                               bf=np.zeros(n, np.uint16)))
            work += [(t, lo, hi) for lo, hi in _runs(ids.size, max(1, n // (4 << 20)))]

        # host work side by side (the C calls release the GIL)
        pool = ThreadPoolExecutor(max(8, min(32, os.cpu_count() or 8)))
        for s in range(1, w.steps + 1):
            list(pool.map(lambda t: W.grad(w, s, t, out=hg[starts[t]:starts[t] + numels[t]]),
                          range(d.n)))
            views = [hg[starts[t]:starts[t] + n] for t, n in enumerate(numels)]
            factor_o, norm_o = oracle.factor(oracle.sumsq(views), w.m, w.max_norm)
            dev_g.copy_(host_g)
            ss.step(grads, params, s)
            torch.cuda.synchronize()
            assert ss.device_error() == 0
            f_g, n_g = float(ss.factor[0].item()), float(ss.norm[0].item())
            assert np.float32(f_g).view(np.uint32) == np.float32(factor_o).view(np.uint32), (s, f_g,
                                                                                          factor_o)
            # the oracle's in-order fp64 sum is within n 2^-53 of the exact sum
            # (textbook bound for positive terms), which bounds the difference
            assert abs(n_g - norm_o) <= max(1e-12, w.numel * 2.0 ** -53) * norm_o, (s, n_g, norm_o)
            # the oracle on every block: each call single-threaded on one run
            # of consecutive blocks of one tensor, the runs side by side
            def run_part(item, s=s, factor=factor_o, views=views):
                t, lo, hi = item
                st = tstate[t]
                sub = {k: v[lo:hi] for k, v in st["blocks"].items()}
                oracle.adam_all(sub, views[t], factor, True, st["mq"], st["vq"], st["msc"][lo:hi],
                                st["vsc"][lo:hi], st["p"], st["bf"], s, hp)
            list(pool.map(run_part, work))

        # copy-in over every tensor, padding untouched, and copy-out
        packed = ss.packed_grad.view(torch.int16)
        for t, n in enumerate(numels):
            o = ss.offsets[t]
            assert torch.equal(packed[o:o + n], grads[t]), f"copy-in differs in tensor {t}"
            assert torch.equal(params[t], ss.packed_bf16.view(torch.int16)[o:o + n]), \
                f"copy-out differs in tensor {t}"
        ends = sorted((o, o + n) for o, n in zip(ss.offsets, numels))
        gaps = [(a[1], b[0]) for a, b in zip(ends, ends[1:]) if b[0] > a[1]]
        for lo, hi in gaps[:50]:
            assert not packed[lo:hi].any(), "padding written"

        # every real element and every block's scales
        msc_g, vsc_g = ss.m_scale.cpu().numpy(), ss.v_scale.cpu().numpy()
        for t, st in enumerate(tstate):
            o, n = ss.offsets[t], numels[t]
            got_p = ss.master[o:o + n].cpu().numpy()
            got_mq = ss.m_state[o:o + n].cpu().numpy()
            got_vq = ss.v_state[o:o + n].cpu().numpy()
            got_bf = ss.packed_bf16.view(torch.int16)[o:o + n].cpu().numpy().view(np.uint16)
            check_master(got_p, st["p"])
            check_codes(got_mq, st["mq"], f"m codes of tensor {t}")
            check_codes(got_vq, st["vq"], f"v codes of tensor {t}")
            assert bit_equal(got_p, st["p"]), f"master of tensor {t} not bit-exact"
            assert np.array_equal(got_mq, st["mq"]), f"m codes of tensor {t} not bit-exact"
            assert np.array_equal(got_vq, st["vq"]), f"v codes of tensor {t} not bit-exact"
            assert bit_equal(got_bf, st["bf"], bf16=True), f"bf16 of tensor {t} not bit-exact"
            assert bit_equal(msc_g[st["ids"]], st["msc"]), f"m scales of tensor {t}"
            assert bit_equal(vsc_g[st["ids"]], st["vsc"]), f"v scales of tensor {t}"

    finally:
        ss.close()
