"""Parity at the full sizes of the four large workloads, in the launch
configuration the benchmark times (ShardStep: pack -> group norm/scale ->
8-bit AdamW -> unpack, every step of the workload's step count).

What the oracle can compute at this size is checked in full; the rest is
sampled:
  - every step: the group norm against the oracle's sum of squares over all
    real gradient elements (within the oracle's own summation error bound,
    n 2^-53 relative) and the scale factor bit for bit;
  - last step: copy-in bit for bit over every tensor (the packed gradient
    against the host gradients, padding still zero) and copy-out bit for bit
    (every parameter tensor against the packed bf16 buffer);
  - sampled quantisation blocks (first, last and random ones of every tensor,
    plus element chunks): the oracle replays each block through every step
    from the same seeded inputs; master, bf16 copy, codes and scales must be
    bit-identical, and in any case within the tolerances (master 1e-6
    relative, codes |d| <= 1 at <= 1e-4 of positions).
"""
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

        rng = np.random.default_rng(1234)
        picks = _sample_blocks(qb, d.n, rng)
        state = {}
        for q in picks:
            t = int(qb["tensor"][q])
            idx = _block_index(qb, q)
            state[q] = dict(p=W.master_init(w, t)[idx - int(off_o[t])].copy(),
                            mq=np.zeros(idx.size, np.int8), vq=np.zeros(idx.size, np.uint8),
                            m_scale=0.0, v_scale=0.0)

        for s in range(1, w.steps + 1):
            for t, n in enumerate(numels):
                W.grad(w, s, t, out=hg[starts[t]:starts[t] + n])
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
            assert np.array_equal(got_bf, want["bf16"]), f"bf16 of block {q}"
            assert float(ss.m_scale[q].item()) == want["m_scale"]
            assert float(ss.v_scale[q].item()) == want["v_scale"]
    finally:
        ss.close()
