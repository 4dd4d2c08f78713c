"""Distributed Muon through the C ABI against the oracle (oracle/muon.py).

Momentum is plain fp32 arithmetic: bit-exact. The orthogonalised update O
goes through the library's tcgen05 products (bf16 operands, fp32 accumulation in an order
the oracle does not reproduce; the oracle's products are exact), so a bf16
result can round to the neighbouring value and Newton-Schulz carries such
flips forward. Tolerance, from that arithmetic: the GPU and the oracle are
two bf16 roundings of one exact iteration, so they lie within 2 d of each
other, d the oracle's own distance from exact arithmetic (the oracle with
exact=True), in Frobenius norm and element by element. Each step's O depends
only on that step's (bit-exact) momentum, so over k steps the masters differ
by at most alpha * sum of the per-step bounds plus fp32 rounding.
"""
import math

import numpy as np
import pytest
import torch

from oracle import muon
from synth import DIST_NORMAL, KIND_GRAD, KIND_PARAM, fill_bf16, fill_f32, key
from synth import workloads as W

pytestmark = pytest.mark.gpu

HP = dict(lr=0.02, momentum=0.95, weight_decay=0.01, eps=1e-7, ns_steps=5, ns_a=3.4445,
          ns_b=-4.7750, ns_c=2.0315)


def _run(specs, m, g_coll, steps, ns_steps=5):
    from fsdp_buffer_layout_gb300 import vsf as V
    from fsdp_buffer_layout_gb300.step import ShardStep, TensorSpec
    hp = dict(HP, ns_steps=ns_steps)
    ss = ShardStep([TensorSpec(*s) for s in specs], m, g_coll)
    try:
        numels = ss.numels
        masters = [fill_f32(key(5, 0, t, KIND_PARAM), DIST_NORMAL, 0.02, 0,
                            np.empty(n, np.float32)) for t, n in enumerate(numels)]
        for t, x in enumerate(masters):
            ss.load_master(t, torch.from_numpy(x).cuda())
        state = {t: dict(M=np.zeros(n, np.float32), p=masters[t].copy(), d_frob=0.0, d_max=0.0)
                 for t, n in enumerate(numels)}
        for s in range(1, steps + 1):
            grads = [fill_bf16(key(5, s, t, KIND_GRAD), DIST_NORMAL, 1e-3, 0,
                               np.empty(n, np.uint16)) for t, n in enumerate(numels)]
            pk = ss.packed_grad.view(torch.int16)
            for t, gr in enumerate(grads):
                pk[ss.offsets[t]:ss.offsets[t] + numels[t]].copy_(
                    torch.from_numpy(gr.view(np.int16)))
            ss.muon_step(V.make_muon_hparams(ns_steps=ns_steps))
            for t, sp in enumerate(specs):
                shape = sp[0]
                if len(shape) < 2:
                    continue
                R, C = shape[-2], shape[-1]
                g32 = (grads[t].astype(np.uint32) << 16).view(np.float32).reshape(-1, R, C)
                M = state[t]["M"].reshape(-1, R, C)
                P = state[t]["p"].reshape(-1, R, C)
                outs = [muon.muon_matrix(g32[e], M[e], P[e], hp) for e in range(g32.shape[0])]
                state[t]["M"] = np.stack([o[0] for o in outs]).ravel()
                state[t]["p"] = np.stack([o[1] for o in outs]).ravel()
                state[t]["O"] = np.stack([o[3] for o in outs]).ravel()
                Oe = np.stack([muon.muon_matrix(g32[e], M[e], P[e], hp, exact=True)[3]
                               for e in range(g32.shape[0])]).ravel()
                diff = state[t]["O"].astype(np.float64) - Oe
                state[t]["d_frob"] += np.linalg.norm(diff)
                state[t]["d_max"] += np.abs(diff).max()
        torch.cuda.synchronize()
        return ss, state, masters
    except Exception:
        ss.close()
        raise


@pytest.mark.parametrize("specs", [
    [((256, 512), W.GRAN_ROWS, 32, 0), ((512,), W.GRAN_ELEM, 0, 0)],
    [((512, 256), W.GRAN_ROWS, 32, 0)],
    [((384, 384), W.GRAN_TILE, 128, 128), ((4, 128, 256), W.GRAN_ROWS, 64, 0)],
    # one shape across tensors (one batched chunk), another shape between them
    [((128, 256), W.GRAN_ROWS, 32, 0), ((96, 64), W.GRAN_ROWS, 32, 0),
     ((2, 128, 256), W.GRAN_ROWS, 64, 0), ((128, 256), W.GRAN_ROWS, 128, 0), ((7,), W.GRAN_ELEM, 0, 0)],
    # 63-element matrices: offsets off the 8-element grid (scalar kernels)
    [((5, 9, 7), W.GRAN_ROWS, 5, 0), ((24, 40), W.GRAN_ROWS, 8, 0)],
    # several 128 x 256 output tiles of the tensor-core kernel, the symmetric
    # products on the tiles at or above the diagonal (wide, tall, batched)
    [((1024, 1536), W.GRAN_ROWS, 32, 0), ((2048, 1024), W.GRAN_ROWS, 64, 0)],
    [((2, 1024, 1024), W.GRAN_ROWS, 128, 0)],
    # ragged tiles: n and k not multiples of the tile (wide, tall)
    [((300, 700), W.GRAN_ROWS, 30, 0), ((1000, 136), W.GRAN_ROWS, 8, 0)],
    # more matrices of one shape than one chunk holds (192)
    [((200, 16, 32), W.GRAN_ROWS, 16, 0), ((3, 32, 16), W.GRAN_ROWS, 32, 0)],
])
def test_muon_matches_oracle(specs):
    ss, state, masters = _run(specs, 4, 128, steps=3)
    try:
        for t, sp in enumerate(specs):
            o, n = ss.offsets[t], ss.numels[t]
            got_p = ss.master[o:o + n].cpu().numpy()
            if len(sp[0]) < 2:
                assert np.array_equal(got_p, masters[t])  # 1-D tensors untouched
                continue
            got_M = ss.momentum[o:o + n].cpu().numpy()
            assert np.array_equal(got_M.view(np.uint32), state[t]["M"].view(np.uint32))
            R, C = sp[0][-2], sp[0][-1]
            alpha = float(np.float32(HP["lr"] * math.sqrt(max(1.0, R / C))))
            ulp = 3 * 2 * float(np.spacing(np.abs(got_p)).max())  # fp32 rounding, 3 steps
            diff = got_p.astype(np.float64) - state[t]["p"].astype(np.float64)
            assert np.abs(diff).max() <= alpha * 2 * state[t]["d_max"] + ulp
            assert np.linalg.norm(diff) <= alpha * 2 * state[t]["d_frob"] + ulp * math.sqrt(n)
            bf = ss.packed_bf16.view(torch.int16)[o:o + n].cpu().numpy().view(np.uint16)
            assert np.array_equal(bf, (muon.bf16_from_f32(got_p).view(np.uint32) >> 16)
                                  .astype(np.uint16))
    finally:
        ss.close()


def test_muon_output_is_orthogonal_band():
    """After one step from zero master, the update (p = -alpha O) has the
    Newton-Schulz singular-value band."""
    from fsdp_buffer_layout_gb300.step import ShardStep, TensorSpec
    ss = ShardStep([TensorSpec((256, 768), W.GRAN_ROWS, 32)], 2, 128)
    try:
        g = fill_bf16(key(9, 1, 0, KIND_GRAD), DIST_NORMAL, 1e-3, 0, np.empty(256 * 768, np.uint16))
        ss.packed_grad.view(torch.int16)[:g.size].copy_(torch.from_numpy(g.view(np.int16)))
        ss.muon_step()
        torch.cuda.synchronize()
        O = -ss.master[:g.size].cpu().numpy().reshape(256, 768) / np.float32(HP["lr"])
        s = np.linalg.svd(O.astype(np.float64), compute_uv=False)
        assert 0.5 <= s.min() and s.max() <= 1.5
    finally:
        ss.close()


@pytest.mark.parametrize("shape", [(256, 512), (512, 256), (3, 128, 192), (1024, 2048),
                                   (2048, 1024), (4096, 4096), (520, 1000)])
def test_muon_update_one_step(shape):
    """Step 1: the update O recovered from the master, (p0 decay - p1) / alpha,
    against the oracle's O. Both are bf16 roundings of the same exact
    Newton-Schulz iteration, so by the triangle inequality they lie within
    twice the oracle's own distance d from exact arithmetic (the oracle run
    with exact=True), in Frobenius norm and element by element. The larger
    shapes span many output tiles (4096 x 4096: 272 of the Gram matrix's 512
    tiles computed, the rest mirrored)."""
    ss, state, masters = _run([(shape, W.GRAN_ROWS, 64, 0)], 2, 128, steps=1)
    try:
        n = ss.numels[0]
        R, C = shape[-2], shape[-1]
        alpha = np.float32(HP["lr"] * math.sqrt(max(1.0, R / C)))
        decay = np.float32(1.0 - HP["lr"] * HP["weight_decay"])
        p1 = ss.master[:n].cpu().numpy().astype(np.float64)
        p0d = (masters[0] * decay).astype(np.float32).astype(np.float64)
        O_gpu = (p0d - p1) / float(alpha)
        g = fill_bf16(key(5, 1, 0, KIND_GRAD), DIST_NORMAL, 1e-3, 0, np.empty(n, np.uint16))
        g32 = (g.astype(np.uint32) << 16).view(np.float32).reshape(-1, R, C)
        zero = np.zeros((R, C), np.float32)
        O, Oe = (np.stack([muon.muon_matrix(g32[e], zero, zero, HP, exact=x)[3]
                           for e in range(g32.shape[0])]).ravel().astype(np.float64)
                 for x in (False, True))
        d_frob, d_max = np.linalg.norm(O - Oe), np.abs(O - Oe).max()
        assert np.linalg.norm(O_gpu - O) <= 2 * d_frob
        assert np.abs(O_gpu - O).max() <= 2 * d_max
        # recovering O from the fp32 master costs far less than a bf16 unit
        assert np.allclose(state[0]["O"], O, rtol=0, atol=0)
    finally:
        ss.close()


def test_two_lanes_are_ordered_on_the_callers_stream():
    """The batched chunks run on two stream lanes (the caller's stream and the
    plan's own). A copy of the bf16 buffer enqueued after the step on the
    caller's stream, and waited for on that stream alone, must see every
    chunk's update, including those of the plan's own lane; and the lanes
    change no arithmetic, so a second plan on the default stream gives the
    same bits."""
    from fsdp_buffer_layout_gb300.step import ShardStep, TensorSpec
    specs = [TensorSpec((2048, 4096), W.GRAN_ROWS, 64), TensorSpec((4096, 1024), W.GRAN_ROWS, 64),
             TensorSpec((2, 1024, 1024), W.GRAN_ROWS, 128)]
    side = torch.cuda.Stream()
    outs = []
    for stream in (side, None):
        ss = ShardStep(specs, 4, 128, stream=stream)
        try:
            assert ss.muon_chunks() == 3
            for t, n in enumerate(ss.numels):
                g = fill_bf16(key(13, 1, t, KIND_GRAD), DIST_NORMAL, 1e-3, 0, np.empty(n, np.uint16))
                o = ss.offsets[t]
                ss.packed_grad.view(torch.int16)[o:o + n].copy_(torch.from_numpy(g.view(np.int16)))
            torch.cuda.synchronize()
            ss.muon_step()
            with torch.cuda.stream(ss.stream):
                snap = ss.packed_bf16.clone()
            ss.stream.synchronize()  # the caller's stream only
            got = snap.view(torch.int16).cpu()
            torch.cuda.synchronize()
            assert torch.equal(got, ss.packed_bf16.view(torch.int16).cpu())
            for t, n in enumerate(ss.numels):  # every tensor was updated
                o = ss.offsets[t]
                assert got[o:o + n].any()
            assert ss.device_error() == 0
            outs.append(got)
        finally:
            ss.close()
    assert torch.equal(outs[0], outs[1])


@pytest.mark.parametrize("ns_steps", [0, 1, 2])
def test_iteration_counts(ns_steps):
    """Newton-Schulz with 0, 1 or 2 iterations instead of 5 (with none, the
    update applies O = X0). Wide, tall and batched matrices, 8-aligned and
    not, three steps, against the oracle. With iterations the bound is the
    one of test_muon_matches_oracle; with none, O = X0 is one bf16 rounding
    of the normalised momentum on both sides, which may differ by one bf16
    unit (2^-8 relative) where the two norms round differently: the masters
    must agree to 2% of how far the three updates moved them."""
    specs = [((256, 512), W.GRAN_ROWS, 32, 0), ((512, 256), W.GRAN_ROWS, 32, 0),
             ((2, 128, 256), W.GRAN_ROWS, 64, 0), ((5, 9, 7), W.GRAN_ROWS, 5, 0)]
    ss, state, masters = _run(specs, 4, 128, steps=3, ns_steps=ns_steps)
    try:
        for t, sp in enumerate(specs):
            o, n = ss.offsets[t], ss.numels[t]
            got_p = ss.master[o:o + n].cpu().numpy()
            got_M = ss.momentum[o:o + n].cpu().numpy()
            assert np.array_equal(got_M.view(np.uint32), state[t]["M"].view(np.uint32))
            R, C = sp[0][-2], sp[0][-1]
            alpha = float(np.float32(HP["lr"] * math.sqrt(max(1.0, R / C))))
            ulp = 3 * 2 * float(np.spacing(np.abs(got_p)).max())
            diff = np.abs(got_p.astype(np.float64) - state[t]["p"].astype(np.float64))
            if ns_steps:
                assert diff.max() <= alpha * 2 * state[t]["d_max"] + ulp
            else:  # a bf16 unit of O is 2^-8 of it: far below the update itself
                decay3 = np.float64(np.float32(1.0 - HP["lr"] * HP["weight_decay"])) ** 3
                moved = np.abs(state[t]["p"].astype(np.float64) - masters[t] * decay3).max()
                assert moved > 0
                assert diff.max() <= 0.02 * moved + ulp
            bf = ss.packed_bf16.view(torch.int16)[o:o + n].cpu().numpy().view(np.uint16)
            assert np.array_equal(bf, (muon.bf16_from_f32(got_p).view(np.uint32) >> 16)
                                  .astype(np.uint16))
        assert ss.device_error() == 0
    finally:
        ss.close()


@pytest.mark.slow
def test_full_llama_layer_one_step():
    """One Muon step of the whole Llama layer (q, k, v, o 4096 x 4096; gate and
    up 11008 x 4096, down 4096 x 11008; two norm vectors) at its own m and
    g_coll, against the oracle matrix by matrix, with the bound of
    test_muon_matches_oracle; the norm vectors stay untouched."""
    w = W.llama_layer()
    specs = [(t.shape, t.gran, t.block_rows, t.tile_cols) for t in w.tensors]
    ss, state, masters = _run(specs, w.m, w.g_coll, steps=1)
    try:
        for t, sp in enumerate(specs):
            o, n = ss.offsets[t], ss.numels[t]
            got_p = ss.master[o:o + n].cpu().numpy()
            if len(sp[0]) < 2:
                assert np.array_equal(got_p, masters[t])
                continue
            R, C = sp[0][-2], sp[0][-1]
            alpha = float(np.float32(HP["lr"] * math.sqrt(max(1.0, R / C))))
            ulp = 2 * float(np.spacing(np.abs(got_p)).max())
            diff = got_p.astype(np.float64) - state[t]["p"].astype(np.float64)
            assert np.abs(diff).max() <= alpha * 2 * state[t]["d_max"] + ulp, t
            assert np.linalg.norm(diff) <= alpha * 2 * state[t]["d_frob"] + ulp * math.sqrt(n), t
        assert ss.device_error() == 0
    finally:
        ss.close()
