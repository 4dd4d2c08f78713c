"""Checkpoint and resume of the optimizer state.

The state is the caller's buffers (master, int8 / uint8 moment codes, their
block scales, bf16 copy). Stopping after step 2, saving to host, restoring
into a fresh ShardStep (new plan, new buffers) and running step 3 must give
the uninterrupted run's step 3 byte for byte; a state taken under another
plan is refused.
"""
import numpy as np
import pytest
import torch

from synth import workloads as W

pytestmark = pytest.mark.gpu


def _shard_step(w, **kw):
    from fsdp_buffer_layout_gb300.step import ShardStep, TensorSpec
    return ShardStep([TensorSpec(t.shape, t.gran, t.block_rows, t.tile_cols) for t in w.tensors],
                     w.m, w.g_coll, max_norm=w.max_norm, **kw)


def _run(ss, w, steps, first=1):
    dev = ss.device
    if first == 1:
        for t in range(len(w.tensors)):
            ss.load_master(t, torch.from_numpy(W.master_init(w, t)).to(dev))
    grads = [torch.empty(n, dtype=torch.int16, device=dev) for n in ss.numels]
    params = [torch.empty(n, dtype=torch.int16, device=dev) for n in ss.numels]
    for s in range(first, first + steps):
        for t, g in enumerate(grads):
            g.copy_(torch.from_numpy(W.grad(w, s, t).view(np.int16)))
        ss.step(grads, params, s)
    torch.cuda.synchronize()
    assert ss.device_error() == 0
    return [p.cpu().numpy() for p in params]


@pytest.mark.parametrize("name", ["tiny", "dsv3_block"])
def test_resume_equals_uninterrupted(name):
    w = W.get(name)
    a = _shard_step(w)
    try:
        want_params = _run(a, w, 3)
        want = a.state_dict()
    finally:
        a.close()
    b = _shard_step(w)
    try:
        _run(b, w, 2)
        sd = b.state_dict()
    finally:
        b.close()
    c = _shard_step(w)
    try:
        c.load_state_dict(sd)
        got_params = _run(c, w, 1, first=3)
        got = c.state_dict()
    finally:
        c.close()
    for k in ("master", "m_state", "v_state", "m_scale", "v_scale", "packed_bf16"):
        assert torch.equal(got[k].view(torch.uint8), want[k].view(torch.uint8)), k
    for x, y in zip(got_params, want_params):
        assert np.array_equal(x, y)


def test_state_from_another_plan_is_refused():
    w = W.tiny()
    a = _shard_step(w)
    try:
        sd = a.state_dict()
    finally:
        a.close()
    b = _shard_step(w.with_(m=2))
    try:
        with pytest.raises(ValueError):
            b.load_state_dict(sd)
    finally:
        b.close()
