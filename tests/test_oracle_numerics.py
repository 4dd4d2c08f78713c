"""Pins of the oracle's copy, norm and AdamW arithmetic against things other
than itself: closed forms, math.fsum, torch.optim.AdamW (CPU, fp32), torch's
bf16 rounding, quantiser properties and the hand-derived fixture
tests/golden/adam8_step1_worked.txt.

Method: "veScale-FSDP: Flexible and High-Performance FSDP at Scale (MLSys
2026)" summary page, 核心方法 > Distributed Buffer (fused group copy / scale)
and 结构感知训练 case study > 8-bit Adam; "FSDP" concept page, 关键观察
(copy-in / copy-out).
"""
import math
import os

import numpy as np
import pytest
import torch

import oracle
import synth
from synth import workloads as W

HP = dict(lr=1e-3, beta1=0.9, beta2=0.999, eps=1e-8, weight_decay=0.01)
GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "adam8_step1_worked.txt")


def f32(x):
    return np.float32(x)


# ---------------------------------------------------------------- copy-in / copy-out

def test_pack_unpack_identity_and_padding_untouched():
    w = W.tiny()
    d = oracle.Desc.from_workload(w)
    S, off = oracle.plan(d, w.m, w.g_coll)
    grads = [W.grad(w, 1, t) for t in range(d.n)]
    packed = oracle.pack(grads, off, w.m * S)
    for t, g in enumerate(grads):
        assert np.array_equal(packed[off[t]:off[t] + g.size], g)
    outs = oracle.unpack(packed, [g.size for g in grads], off)
    for a, b in zip(outs, grads):
        assert np.array_equal(a, b)
    real = np.zeros(w.m * S, bool)
    for t, g in enumerate(grads):
        real[off[t]:off[t] + g.size] = True
    assert not packed[~real].any()


def test_pack_fp32():
    a = np.arange(10, dtype=np.float32)
    b = -np.arange(3, dtype=np.float32)
    packed = oracle.pack([a, b], [0, 16], 32)
    assert np.array_equal(packed[:10], a) and np.array_equal(packed[16:19], b)


# ---------------------------------------------------------------- norm and scale

def test_sumsq_constant_closed_form():
    c = 2.0 ** -9
    bits = np.array([c], np.float32).view(np.uint32)[0] >> 16
    ts = [np.full(1000, bits, np.uint16), np.full(24, bits | 0x8000, np.uint16)]
    assert oracle.sumsq(ts) == 1024 * c * c


def test_sumsq_matches_fsum():
    w = W.tiny()
    grads = [W.grad(w, 1, t) for t in range(len(w.tensors))]
    n = sum(g.size for g in grads)
    bound = n * 2.0 ** -53  # textbook bound of a recursive fp64 sum of positive terms
    got = oracle.sumsq(grads)
    want = math.fsum(float(x) ** 2 for g in grads for x in synth.bf16_to_f32(g))
    assert abs(got - want) <= bound * want
    g32 = [W.grad_f32(w, 1, t) for t in range(len(w.tensors))]
    got32 = oracle.sumsq(g32)
    want32 = math.fsum(float(x) ** 2 for g in g32 for x in g)
    assert abs(got32 - want32) <= bound * want32


def test_factor_no_clip_is_exact_inverse_world():
    for world in (1, 4, 8, 64, 1024, 3):
        f, norm = oracle.factor(1234.5, world, math.inf)
        assert f == float(np.float32(1.0 / world))
        assert norm == math.sqrt(1234.5) / world


def test_factor_clip_closed_form():
    # sumsq = 400 -> sqrt = 20 -> norm over world 4 = 5; c = 1/(5 + 1e-6)
    f, norm = oracle.factor(400.0, 4, 1.0)
    assert norm == 5.0
    assert f == float(np.float32((1.0 / (5.0 + 1e-6)) / 4.0))
    f2, _ = oracle.factor(400.0, 4, 10.0)  # norm under the limit: no clipping
    assert f2 == 0.25


# ---------------------------------------------------------------- bf16 rounding

def test_bf16_round_matches_torch():
    rng = np.random.default_rng(0)
    x = np.concatenate([rng.standard_normal(20000).astype(np.float32) * 0.02,
                        np.array([1 + 2 ** -8, 1 + 3 * 2 ** -8, -(1 + 2 ** -8), 3.4e38, -0.0,
                                  1e-40, np.inf, -np.inf], np.float32)])
    want = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    got = np.array([oracle.bf16_round(float(v)) for v in x], np.uint16)
    assert np.array_equal(got, want)


def test_bf16_round_nan_is_nan():
    """IEEE 754 makes a converted NaN a NaN, whatever its bits (torch's own
    scalar and vectorised conversions disagree on them), so only the class is
    pinned: exponent all ones and a nonzero fraction, for quiet, signalling
    and negative NaNs alike."""
    for bits in (0x7FC00000, 0xFFC00000, 0x7F800001, 0xFF812345, 0x7FFFFFFF):
        f = float(np.array([bits], np.uint32).view(np.float32)[0])
        h = oracle.bf16_round(f)
        assert (h & 0x7F80) == 0x7F80 and (h & 0x007F) != 0, hex(h)


# ---------------------------------------------------------------- AdamW, fp32 state

def adam_fp32_steps(g_list, p0, factor):
    st = dict(p=p0.copy(), m=np.zeros_like(p0), v=np.zeros_like(p0))
    for t, g in enumerate(g_list, start=1):
        st = oracle.adam_block(g, False, factor, st, t, HP)
    return st


def test_first_step_closed_form():
    """Step 1 with zero state: p1 = p (1 - lr wd) - lr g / (|g| + eps)."""
    w = W.tiny()
    g = W.grad(w, 1, 0)
    p0 = W.master_init(w, 0)
    factor = 0.25
    st = adam_fp32_steps([g], p0, factor)
    gs = factor * synth.bf16_to_f32(g).astype(np.float64)
    want = p0.astype(np.float64) * (1 - HP["lr"] * HP["weight_decay"]) \
        - HP["lr"] * gs / (np.abs(gs) + HP["eps"])
    err = np.abs(st["p"].astype(np.float64) - want)
    assert np.all(err <= 1e-6 * (np.abs(want) + HP["lr"]))
    assert np.abs(st["p"] - p0).max() > 5e-4  # the update really happened


def test_zero_grad_step_is_pure_decay():
    p0 = np.array([0.5, -0.25, 0.0, 1e-3], np.float32)
    g = np.zeros(4, np.uint16)
    st = adam_fp32_steps([g], p0, 1.0)
    assert np.array_equal(st["p"], p0 * np.float32(1 - 1e-5))


def test_matches_torch_adamw_ten_steps():
    """Textbook AdamW (torch.optim.AdamW, CPU fp32, single-tensor path)."""
    w = W.tiny()
    n = 4096
    p0 = W.master_init(w, 0)[:n].copy()
    factor = np.float32(0.25)
    gs = [W.grad(w, s, 0)[:n].copy() for s in range(1, 11)]
    st = dict(p=p0.copy(), m=np.zeros(n, np.float32), v=np.zeros(n, np.float32))
    prm = torch.nn.Parameter(torch.from_numpy(p0.copy()))
    opt = torch.optim.AdamW([prm], lr=HP["lr"], betas=(HP["beta1"], HP["beta2"]), eps=HP["eps"],
                            weight_decay=HP["weight_decay"], foreach=False, fused=False)
    for t, g in enumerate(gs, start=1):
        st = oracle.adam_block(g, False, float(factor), st, t, HP)
        prm.grad = torch.from_numpy(synth.bf16_to_f32(g) * factor)
        opt.step()
        ref = prm.detach().numpy().astype(np.float64)
        err = np.abs(st["p"].astype(np.float64) - ref)
        # torch rounds in another order (lerp for m, two divisions); a few ulps
        # of the master accumulate over the steps. A wrong term or sign shows
        # up at the size of an update (lr = 1e-3), four orders above this bound.
        assert np.all(err <= 1e-6 * np.abs(ref) + 1e-7), (t, err.max())
        sref = opt.state[prm]
        # torch writes m as a lerp, so moments agree to rounding of the largest one
        for mine, theirs in ((st["m"], sref["exp_avg"].numpy()),
                             (st["v"], sref["exp_avg_sq"].numpy())):
            assert np.abs(mine - theirs).max() <= 1e-6 * np.abs(theirs).max()


# ---------------------------------------------------------------- quantiser

def test_quantizer_properties():
    rng = np.random.default_rng(3)
    for trial in range(50):
        x = (rng.standard_normal(int(rng.integers(1, 600))) * 10.0 ** rng.integers(-9, 2)).astype(
            np.float32)
        c, s, dq = oracle.quantize_m(x)
        assert s == np.abs(x).max()
        assert np.all(np.abs(c.astype(int)) <= 127)
        assert np.abs(c[np.argmax(np.abs(x))]) == 127
        assert np.all(np.abs(dq.astype(np.float64) - x) <= s / 254 * (1 + 1e-5))
        c2, s2, _ = oracle.quantize_m(dq)
        assert np.array_equal(c2, c)  # idempotent on its own grid
        v = np.abs(x) ** 2
        cv, sv, dv = oracle.quantize_v(v)
        assert sv == v.max() and cv[np.argmax(v)] == 255
        assert np.all(np.abs(dv.astype(np.float64) - v) <= sv / 510 * (1 + 1e-5))
        cv2, _, _ = oracle.quantize_v(dv)
        assert np.array_equal(cv2, cv)


def test_quantizer_tiny_scale_stays_symmetric():
    """A block scale below 127 / FLT_MAX (about 3.7e-37) makes 127 / scale
    overflow to infinity: every nonzero element then saturates. The m codes
    must stay in the symmetric range, +-127 (a clamp at -128 would give
    negative elements code -128, which dequantises above the absmax), zeros
    stay 0, and no dequantised value exceeds the scale."""
    s = np.float32(127.0 * 2.0 ** -130)          # normal, and 127 / s = 2^130 > FLT_MAX
    with np.errstate(over="ignore"):
        assert np.float32(127.0) / s == np.inf
    x = np.array([s, -s, -s / 2, s / 3, 0.0, -2.0 ** -149, 2.0 ** -140], np.float32)
    c, scale, dq = oracle.quantize_m(x)
    assert scale == s
    assert list(c) == [127, -127, -127, 127, 0, -127, 127]
    assert np.all(np.abs(dq) <= s)
    assert np.abs(dq).max() == s                   # 127 * (s / 127) is exact here
    # the same through the v quantiser: 255 / scale overflows, all saturate to 255
    v = np.abs(x)
    cv, sv, dv = oracle.quantize_v(v)
    assert list(cv) == [255, 255, 255, 255, 0, 255, 255] and sv == s
    assert np.all(dv <= np.float32(255.0) * (s / np.float32(255.0)))


def test_quantizer_zero_block_and_ties():
    c, s, dq = oracle.quantize_m(np.zeros(7, np.float32))
    assert s == 0 and not c.any() and not dq.any()
    cv, sv, dv = oracle.quantize_v(np.zeros(7, np.float32))
    assert sv == 0 and not cv.any() and not dv.any()
    # 127 * [1, 1/254, 3/254] = [127, 0.5, 1.5]: exact halves round to even (0, 2)
    x = np.array([254.0, 1.0, 3.0], np.float32)
    c, s, _ = oracle.quantize_m(x)
    assert list(c) == [127, 0, 2]


def load_worked():
    rows = {}
    for line in open(GOLDEN):
        if line.startswith("#") or not line.strip():
            continue
        k, *vals = line.split()
        rows[k] = vals
    return rows


def test_worked_example_step1():
    fx = load_worked()
    g = np.array([int(v, 16) for v in fx["g_bf16"]], np.uint16)
    p0 = np.array([0.02, -0.02, 0.0, 0.5], np.float32)
    st = dict(p=p0.copy(), mq=np.zeros(4, np.int8), vq=np.zeros(4, np.uint8),
              m_scale=0.0, v_scale=0.0)
    out = oracle.adam_block(g, True, 1.0, st, 1, HP)
    assert list(out["mq"]) == [int(v) for v in fx["m_codes"]]
    assert list(out["vq"]) == [int(v) for v in fx["v_codes"]]
    assert out["m_scale"] == float(np.float32(np.float32(0.1) * np.float32(2.0 ** -10)))
    assert out["v_scale"] == float(np.float32(np.float32(0.001) * np.float32(2.0 ** -20)))
    gs = synth.bf16_to_f32(g).astype(np.float64)
    want = p0 * (1 - 1e-5) - 1e-3 * gs / (np.abs(gs) + 1e-8)
    assert np.all(np.abs(out["p"] - want) <= 1e-6 * (np.abs(want) + 1e-3))


def test_quantized_step1_master_equals_fp32_step1():
    """At step 1 the update only sees fresh moments: the 8-bit and fp32-state
    masters agree bit for bit."""
    w = W.llama_layer()
    g = W.grad(w, 1, 0, 0, 4096 * 32)
    p0 = W.master_init(w, 0, 0, 4096 * 32)
    q = oracle.adam_block(g, True, 0.125, dict(p=p0, mq=np.zeros(g.size, np.int8),
                                                 vq=np.zeros(g.size, np.uint8),
                                                 m_scale=0.0, v_scale=0.0), 1, HP)
    f = oracle.adam_block(g, False, 0.125, dict(p=p0, m=np.zeros(g.size, np.float32),
                                                  v=np.zeros(g.size, np.float32)), 1, HP)
    assert np.array_equal(q["p"], f["p"]) and np.array_equal(q["bf16"], f["bf16"])
    cm, sm, _ = oracle.quantize_m(f["m"])
    cv, sv, _ = oracle.quantize_v(f["v"])
    assert np.array_equal(q["mq"], cm) and np.array_equal(q["vq"], cv)
    assert (q["m_scale"], q["v_scale"]) == (sm, sv)


def test_quantized_step_is_dequant_update_requant():
    """Requantisation follows the update, with the new block scale."""
    w = W.tiny()
    n = 8192
    rng = np.random.default_rng(5)
    mq = rng.integers(-127, 128, n).astype(np.int8)
    vq = rng.integers(0, 256, n).astype(np.uint8)
    ms, vs = 3e-5, 2e-9
    p0 = W.master_init(w, 0, 0, n)
    g = W.grad(w, 4, 0, 0, n)
    q = oracle.adam_block(g, True, 0.25, dict(p=p0, mq=mq, vq=vq, m_scale=ms, v_scale=vs), 4, HP)
    m_deq = mq.astype(np.float32) * np.float32(np.float32(ms) / np.float32(127))
    v_deq = vq.astype(np.float32) * np.float32(np.float32(vs) / np.float32(255))
    f = oracle.adam_block(g, False, 0.25, dict(p=p0, m=m_deq, v=v_deq), 4, HP)
    assert np.array_equal(q["p"], f["p"])
    cm, sm, _ = oracle.quantize_m(f["m"])
    cv, sv, _ = oracle.quantize_v(f["v"])
    assert np.array_equal(q["mq"], cm) and np.array_equal(q["vq"], cv)
    assert (q["m_scale"], q["v_scale"]) == (sm, sv)


def test_adam_all_matches_blockwise():
    w = W.tiny()
    d = oracle.Desc.from_workload(w)
    S, off = oracle.plan(d, w.m, w.g_coll)
    qb = oracle.qblocks(d, w.g_coll, off)
    total = w.m * S
    grads = [W.grad(w, 1, t) for t in range(d.n)]
    packed = oracle.pack(grads, off, total)
    master = oracle.pack([W.master_init(w, t) for t in range(d.n)], off, total)
    mq, vq = np.zeros(total, np.int8), np.zeros(total, np.uint8)
    nq = len(qb["base"])
    ms, vs = np.zeros(nq, np.float32), np.zeros(nq, np.float32)
    bf = np.zeros(total, np.uint16)
    oracle.adam_all(qb, packed, 0.25, True, mq, vq, ms, vs, master, bf, 1, HP)
    # one TILE block (tensor 2, first tile) recomputed on its own
    q = int(np.nonzero(qb["tensor"] == 2)[0][1])
    r, c, s, b = (int(qb[k][q]) for k in ("nrows", "ncols", "stride", "base"))
    idx = (b + np.arange(r)[:, None] * s + np.arange(c)[None, :]).ravel()
    g = packed[idx]
    p0 = oracle.pack([W.master_init(w, t) for t in range(d.n)], off, total)[idx]
    one = oracle.adam_block(g, True, 0.25, dict(p=p0, mq=np.zeros(idx.size, np.int8),
                                                  vq=np.zeros(idx.size, np.uint8),
                                                  m_scale=0.0, v_scale=0.0), 1, HP)
    assert np.array_equal(master[idx], one["p"]) and np.array_equal(mq[idx], one["mq"])
    assert ms[q] == one["m_scale"]


# ---------------------------------------------------------------- fused group ops

def test_group_ops_closed_forms():
    """zero -> 0; x + (-x) -> 0; scale by 2 is exact; padding untouched."""
    rng = np.random.default_rng(9)
    x = (rng.standard_normal(64) * 1e-3).astype(np.float32)
    buf = np.full(80, 7.0, np.float32)
    buf[3:3 + 64] = x
    oracle.group_op(1, [64], [3], buf, alpha=2.0)
    assert np.array_equal(buf[3:67], x * np.float32(2)) and buf[0] == 7 and buf[70] == 7
    neg = np.zeros(80, np.float32)
    neg[3:67] = -x * 2
    oracle.group_op(2, [64], [3], buf, neg)
    assert not buf[3:67].any() and buf[0] == 7
    buf[3:67] = x
    oracle.group_op(0, [64], [3], buf)
    assert not buf[3:67].any() and buf[67:].tolist() == [7.0] * 13


def test_group_add_bf16_matches_numpy_and_torch_rounding():
    """bf16 accumulation: the fp32 sum (numpy) rounded by torch's bf16 conversion."""
    w = W.tiny()
    a = W.grad(w, 1, 0, 0, 4096)
    b = W.grad(w, 2, 0, 0, 4096)
    dst = np.concatenate([np.zeros(5, np.uint16), a, np.zeros(3, np.uint16)])
    src = np.concatenate([np.zeros(5, np.uint16), b, np.zeros(3, np.uint16)])
    oracle.group_op(2, [4096], [5], dst, src)
    s32 = synth.bf16_to_f32(a) + synth.bf16_to_f32(b)
    want = torch.from_numpy(s32).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(dst[5:5 + 4096], want)
    # fp32 destination accumulating bf16: exact fp32 sums
    acc = np.zeros(4096, np.float32)
    oracle.group_op(2, [4096], [0], acc, a)
    oracle.group_op(2, [4096], [0], acc, b)
    assert np.array_equal(acc, s32)


def test_blocks_are_independent_across_calls():
    """The 8-bit step of one quantisation block reads and writes only that
    block's elements and its own two scales ([VSF] case study › 8-bit Adam:
    block-wise quantisation, no block crosses a rank), so running a tensor's
    blocks as several runs of consecutive blocks, in any order, gives the
    same state bit for bit as one call over all of them. The full-size GPU
    parity relies on this to replay large tensors on host threads."""
    w = W.tiny()
    d = oracle.Desc.from_workload(w)
    S, off = oracle.plan(d, w.m, w.g_coll)
    qb = oracle.qblocks(d, w.g_coll, off)
    hp = oracle.hparams(w)
    t = int(np.argmax([x.numel for x in w.tensors]))
    ids = np.nonzero(qb["tensor"] == t)[0]
    blocks = {k: np.ascontiguousarray(qb[k][ids]) for k in ("base", "nrows", "ncols", "stride")}
    blocks["base"] = blocks["base"] - int(off[t])
    n = w.tensors[t].numel
    assert ids.size >= 8

    def fresh():
        return dict(p=W.master_init(w, t).copy(), mq=np.zeros(n, np.int8), vq=np.zeros(n, np.uint8),
                    msc=np.zeros(ids.size, np.float32), vsc=np.zeros(ids.size, np.float32),
                    bf=np.zeros(n, np.uint16))

    whole, parts = fresh(), fresh()
    runs = [(0, 3), (3, 4), (4, ids.size)]
    for s in range(1, 4):
        g = W.grad(w, s, t)
        oracle.adam_all(blocks, g, 0.25, True, whole["mq"], whole["vq"], whole["msc"], whole["vsc"],
                        whole["p"], whole["bf"], s, hp)
        for lo, hi in reversed(runs):
            sub = {k: v[lo:hi] for k, v in blocks.items()}
            oracle.adam_all(sub, g, 0.25, True, parts["mq"], parts["vq"], parts["msc"][lo:hi],
                            parts["vsc"][lo:hi], parts["p"], parts["bf"], s, hp)
    for k in whole:
        assert np.array_equal(whole[k].view(np.uint8), parts[k].view(np.uint8)), k
