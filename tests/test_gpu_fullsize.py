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
The optimizer state:
  - Llama layer and DSv3 block: in full. The oracle runs every quantisation
    block through every step (per tensor, on the tensor's real elements),
    and the final master, m and v codes, m and v scales and bf16 copy of
    every real element must be bit-identical (NaNs by class), and in any
    case within the tolerances (master 1e-6 relative, codes |d| <= 1 at
    <= 1e-4 of positions);
  - MoE layer and 1.3B model: sampled quantisation blocks (first, last and
    random ones of every tensor, plus element chunks) replayed by the oracle
    through every step, under the same bar (host time: the oracle runs
    single-threaded at about 80 M elements per second).
"""
from concurrent.futures import ThreadPoolExecutor

import numpy as np
import pytest
import torch

import oracle
from synth import workloads as W

from gpu_harness import bit_equal, check_codes, check_master

pytestmark = [pytest.mark.gpu, pytest.mark.slow]

HP = dict(lr=1e-3, beta1=0.9, beta2=0.999, eps=1e-8, weight_decay=0.01)


def _sample_blocks(qb, n_tensors, rng):
    picks = []
    for t in range(n_tensors):
        ids = np.nonzero(qb["tensor"] == t)[0]
        chosen = {int(ids[0]), int(ids[-1])}
        if ids.size > 2:
            chosen |= {int(x) for x in rng.choice(ids[1:-1], size=min(2, ids.size - 2),
                                                  replace=False)}
        picks += sorted(chosen)
    return picks


def _block_index(qb, q):
    base, nr, nc, st = (int(qb[k][q]) for k in ("base", "nrows", "ncols", "stride"))
    return (base + np.arange(nr, dtype=np.int64)[:, None] * st
            + np.arange(nc, dtype=np.int64)[None, :]).ravel()


def _tensor_blocks(qb, off_o, t):
    """The quantisation blocks of tensor t, re-based to the tensor's own
    element 0 (so that the oracle can run them on per-tensor arrays), and
    their indices in the whole plan's block table."""
    ids = np.nonzero(qb["tensor"] == t)[0]
    blocks = {k: np.ascontiguousarray(qb[k][ids]) for k in ("base", "nrows", "ncols", "stride")}
    blocks["base"] = blocks["base"] - int(off_o[t])
    return blocks, ids


@pytest.mark.parametrize("name,full", [("llama_layer", True), ("moe_layer", False),
                                       ("dsv3_block", True), ("llama_1p3b", False)])
def test_fullsize_workload(name, full):
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

        rng = np.random.default_rng(1234)
        picks = [] if full else _sample_blocks(qb, d.n, rng)
        hp = oracle.hparams(w)
        tstate = []  # full mode: the oracle's state of every tensor, tensor-local
        if full:
            for t in range(d.n):
                blocks, ids = _tensor_blocks(qb, off_o, t)
                n = numels[t]
                tstate.append(dict(blocks=blocks, ids=ids, p=W.master_init(w, t).copy(),
                                   mq=np.zeros(n, np.int8), vq=np.zeros(n, np.uint8),
                                   msc=np.zeros(ids.size, np.float32),
                                   vsc=np.zeros(ids.size, np.float32),
                                   bf=np.zeros(n, np.uint16)))
        state = {}
        for q in picks:
            t = int(qb["tensor"][q])
            idx = _block_index(qb, q)
            state[q] = dict(p=W.master_init(w, t)[idx - int(off_o[t])].copy(),
                            mq=np.zeros(idx.size, np.int8), vq=np.zeros(idx.size, np.uint8),
                            m_scale=0.0, v_scale=0.0)

        pool = ThreadPoolExecutor(8)  # host work per tensor (the C calls release the GIL)
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
            for q in picks:
                t = int(qb["tensor"][q])
                idx = _block_index(qb, q)
                g = hg[starts[t]:starts[t] + numels[t]][idx - int(off_o[t])]
                state[q] = oracle.adam_block(np.ascontiguousarray(g), True, factor_o, state[q], s,
                                             HP)
            # the oracle on every tensor (each call single-threaded, tensors side by side)
            def run_tensor(t, s=s, factor=factor_o, views=views):
                st = tstate[t]
                oracle.adam_all(st["blocks"], np.ascontiguousarray(views[t]), factor, True,
                                st["mq"], st["vq"], st["msc"], st["vsc"], st["p"], st["bf"], s, hp)
            list(pool.map(run_tensor, range(len(tstate))))

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

        # full mode: every real element and every block's scales
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

        # sampled blocks against the oracle's replay
        for q in picks:
            idx = torch.from_numpy(_block_index(qb, q)).to(dev)
            want = state[q]
            got_p = ss.master[idx].cpu().numpy()
            got_mq = ss.m_state[idx].cpu().numpy()
            got_vq = ss.v_state[idx].cpu().numpy()
            got_bf = ss.packed_bf16.view(torch.int16)[idx].cpu().numpy().view(np.uint16)
            check_master(got_p, want["p"])
            check_codes(got_mq, want["mq"], f"m codes of block {q}")
            check_codes(got_vq, want["vq"], f"v codes of block {q}")
            assert bit_equal(got_p, want["p"]), f"master of block {q} not bit-exact"
            assert np.array_equal(got_mq, want["mq"]) and np.array_equal(got_vq, want["vq"])
            assert bit_equal(got_bf, want["bf16"], bf16=True), f"bf16 of block {q}"
            assert float(ss.m_scale[q].item()) == want["m_scale"]
            assert float(ss.v_scale[q].item()) == want["v_scale"]
    finally:
        ss.close()
