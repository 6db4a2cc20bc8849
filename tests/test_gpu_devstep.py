"""GPU parity of the device-resident step (fp8_adam_step_dev,
fp8_cast_adamw_step_dev): lr, inv_loss_scale and the step count are read from
device memory at run or graph-replay time.  Lock-step against the oracle with
a changing learning rate and loss scale, equality with the host-scalar calls,
CUDA-graph replays across steps, the GradScaler skip (the step count does
not advance) and empty lists."""
import dataclasses

import numpy as np
import pytest
import torch

import oracle
import synth
from harness import GpuState, fresh_states, oracle_cast, set_grads

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def bo():
    import bit_optimizer_gb300 as bo
    return bo


@pytest.fixture
def stream(bo):
    import gc
    s = torch.cuda.Stream()
    yield s
    gc.collect()
    torch.cuda.synchronize()
    bo.release_stream(s)


def schedule(t):
    """lr and inv_loss_scale of step t: both change every step."""
    return 1e-3 * (1.0 + 0.37 * t), 2.0 ** -(14 + t % 3)


@pytest.mark.parametrize("level,l2,scaled_v", [("O2", False, False),
                                               ("O3", False, True),
                                               ("O2", True, False)])
def test_dev_step_lock_step_with_oracle(bo, level, l2, scaled_v):
    mk = synth.o2_350m if level == "O2" else synth.o3_1p3b
    wl = dataclasses.replace(mk(n_layer=1, d=64, ffn=256, vocab=333, ctx=40),
                             inf_site=None)
    weights = wl.weights()
    states = fresh_states(weights, level == "O3", scaled_v=scaled_v)
    gs = GpuState(states)
    st = bo.StepState(device="cuda")
    found = torch.full((1,), 7, dtype=torch.int32, device="cuda")
    for t in range(1, 5):
        lr, ils = schedule(t)
        codes, _, scales = oracle_cast(wl.grads(t), oracle.E4M3)
        set_grads(states, codes, scales)
        for i, c in enumerate(codes):
            gs.g[i].copy_(torch.from_numpy(c))
        gs.g_scale[:len(scales)].copy_(torch.from_numpy(scales))
        st.lr.fill_(lr)
        st.inv_loss_scale.fill_(ils)
        gs.plan.step_dev(st, wl.beta1, wl.beta2, wl.eps, wl.wd, l2=l2,
                         found_inf_dev=found)
        assert oracle.adamw_step(states, lr, wl.beta1, wl.beta2, wl.eps, wl.wd, t,
                                 ils, l2=l2) == 0
        torch.cuda.synchronize()
        assert found.item() == 0
        assert st.step.item() == t
        rates = gs.compare(states)
        assert min(rates.values()) == 1.0, rates


def _host_and_dev_pair(bo, wl, **kw):
    """Two optimizers over equal copies of the weights: host scalars, and a
    capturable one."""
    w = wl.weights()
    p_host = [x.cuda() for x in w]
    p_dev = [x.cuda() for x in w]
    host = bo.Fp8AdamW(p_host, lr=wl.lr, betas=(wl.beta1, wl.beta2), eps=wl.eps,
                       weight_decay=wl.wd, **kw)
    dev = bo.Fp8AdamW(p_dev, lr=wl.lr, betas=(wl.beta1, wl.beta2), eps=wl.eps,
                      weight_decay=wl.wd, capturable=True, **kw)
    return host, dev, p_host, p_dev


def _assert_same(host, dev, p_host, p_dev):
    for a, b in zip(p_host, p_dev):
        assert torch.equal(a, b)
    for a, b in zip(host.m + host.v, dev.m + dev.v):
        assert torch.equal(a, b)
    assert torch.equal(host.m_scale, dev.m_scale)
    if host.w8 is not None:
        for a, b in zip(host.w8, dev.w8):
            assert torch.equal(a, b)
        assert torch.equal(host.w8_scale, dev.w8_scale)
    if host.v_bound is not None:
        assert torch.equal(host.v_bound, dev.v_bound)


@pytest.mark.parametrize("kw", [dict(level="O2"),
                                dict(level="O3", scaled_v=True),
                                dict(level="O2", l2=True),
                                dict(level="O2", fused=False),
                                dict(level="O2", max_grad_norm=0.05),
                                dict(level="O3", l2=True, max_grad_norm=0.05)])
def test_dev_step_equals_host_step(bo, kw):
    wl = dataclasses.replace(
        synth.o2_6p7b_tail(n_layer=1, d=64, ffn=256, vocab=500, ctx=64, n_tail=20),
        inf_site=None)
    host, dev, p_host, p_dev = _host_and_dev_pair(bo, wl, **kw)
    grads = [torch.empty(n, dtype=torch.bfloat16, device="cuda") for n in wl.numels]
    for t in range(1, 5):
        lr, ils = schedule(t)
        for i, g in enumerate(grads):
            g.copy_(wl.grad(i, t, "cuda"))
        host.lr = lr
        assert host.step(grads, ils) == 0
        dev.set_lr(lr)
        dev.state.inv_loss_scale.fill_(ils)
        assert dev.step(grads) is None
        torch.cuda.synchronize()
        assert dev.state.step.item() == t == host.step_count
        _assert_same(host, dev, p_host, p_dev)
        if "max_grad_norm" in kw:
            # the same norm, as a float on the device
            assert dev.grad_norm_dev.item() == np.float32(host.last_grad_norm)


def test_dev_step_graph_replays_follow_the_schedule(bo, stream):
    """One captured fused step, replayed for steps 2..6 with a new lr, loss
    scale and gradients each time, gives the host-scalar steps' bytes."""
    wl = dataclasses.replace(
        synth.o3_1p3b(n_layer=1, d=64, ffn=256, vocab=300, ctx=32), inf_site=None)
    s = stream
    with torch.cuda.stream(s):
        host, dev, p_host, p_dev = _host_and_dev_pair(bo, wl, level="O3")
        grads = [torch.empty(n, dtype=torch.bfloat16, device="cuda")
                 for n in wl.numels]
        flag = torch.full((1,), 7, dtype=torch.int32, device="cuda")
        lr, ils = schedule(1)
        for i, g in enumerate(grads):
            g.copy_(wl.grad(i, 1, "cuda"))
        dev.set_lr(lr)
        dev.state.inv_loss_scale.fill_(ils)
        dev.step(grads, found_inf_dev=flag, stream=s)        # step 1, direct
    s.synchronize()
    host.lr = lr
    assert host.step(grads, ils) == 0
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        dev.step(grads, found_inf_dev=flag, stream=s)
    torch.cuda.synchronize()
    assert dev.state.step.item() == 1          # capture runs nothing
    for t in range(2, 7):
        lr, ils = schedule(t)
        with torch.cuda.stream(s):
            for i, x in enumerate(grads):
                x.copy_(wl.grad(i, t, "cuda"))
            dev.set_lr(lr)
            dev.state.inv_loss_scale.fill_(ils)
            g.replay()
        s.synchronize()
        host.lr = lr
        assert host.step(grads, ils) == 0
        torch.cuda.synchronize()
        assert flag.item() == 0 and dev.state.step.item() == t
        _assert_same(host, dev, p_host, p_dev)


@pytest.mark.parametrize("fused", [True, False])
def test_dev_step_skip_keeps_state_and_step_count(bo, fused):
    wl = dataclasses.replace(synth.o2_350m(n_layer=1, d=64, ffn=256, vocab=300,
                                           ctx=32), inf_site=None)
    host, dev, p_host, p_dev = _host_and_dev_pair(bo, wl, fused=fused)
    grads = [torch.empty(n, dtype=torch.bfloat16, device="cuda") for n in wl.numels]
    for i, g in enumerate(grads):
        g.copy_(wl.grad(i, 1, "cuda"))
    flag = torch.full((1,), 7, dtype=torch.int32, device="cuda")
    dev.step(grads, found_inf_dev=flag)
    assert host.step(grads) == 0
    torch.cuda.synchronize()
    assert flag.item() == 0 and dev.state.step.item() == 1
    grads[3].view(-1)[5] = float("inf")
    before = [t.clone() for t in p_dev + dev.m + dev.v] + [dev.m_scale.clone()]
    dev.step(grads, found_inf_dev=flag)
    torch.cuda.synchronize()
    assert flag.item() == 1
    assert dev.state.step.item() == 1          # a skipped step does not count
    after = [t for t in p_dev + dev.m + dev.v] + [dev.m_scale]
    for a, b in zip(before, after):
        assert torch.equal(a, b)
    # the next good step is step 2 on both sides
    for i, g in enumerate(grads):
        g.copy_(wl.grad(i, 2, "cuda"))
    dev.step(grads, found_inf_dev=flag)
    assert host.step(grads) == 0
    torch.cuda.synchronize()
    assert flag.item() == 0 and dev.state.step.item() == 2 == host.step_count
    _assert_same(host, dev, p_host, p_dev)


def test_dev_step_empty_lists_advance_the_step(bo):
    st = bo.StepState(device="cuda", step=41)
    flag = torch.full((1,), 7, dtype=torch.int32, device="cuda")
    empty = bo.AdamWPlan([], torch.ones(1, device="cuda"), [],
                         torch.ones(1, device="cuda"), [], [])
    empty.step_dev(st, 0.9, 0.999, 1e-8, 0.0, found_inf_dev=flag)
    torch.cuda.synchronize()
    assert st.step.item() == 42 and flag.item() == 0
    # a list of empty tensors has no chunks: the step is still taken
    z = [torch.empty(0, dtype=torch.float16, device="cuda")]
    opt = bo.Fp8AdamW(z, capturable=True)
    opt.step([torch.empty(0, dtype=torch.bfloat16, device="cuda")],
             found_inf_dev=flag)
    torch.cuda.synchronize()
    assert opt.state.step.item() == 1 and flag.item() == 0


def test_dev_step_state_dict_round_trip(bo):
    wl = dataclasses.replace(synth.o2_350m(n_layer=1, d=64, ffn=256, vocab=300,
                                           ctx=32), inf_site=None)
    p = [x.cuda() for x in wl.weights()]
    opt = bo.Fp8AdamW(p, capturable=True)
    grads = [g.cuda() for g in wl.grads(1)]
    opt.set_lr(3e-4)
    opt.step(grads)
    opt.step(grads)
    d = opt.state_dict()
    assert d["step"] == 2 and d["hparams"][0] == np.float32(3e-4)
    opt2 = bo.Fp8AdamW([x.clone() for x in p], capturable=True)
    opt2.load_state_dict(d)
    assert opt2.state.step.item() == 2
    assert opt2.state.lr.item() == np.float32(3e-4)


def test_clipped_dev_step_graph_replays(bo, stream):
    """A captured clipped fused step (the norm and its coefficient depend on
    the replayed inv_loss_scale) follows the host-scalar clipped steps."""
    wl = dataclasses.replace(
        synth.o2_350m(n_layer=1, d=64, ffn=256, vocab=300, ctx=32), inf_site=None)
    s = stream
    with torch.cuda.stream(s):
        host, dev, p_host, p_dev = _host_and_dev_pair(bo, wl, max_grad_norm=0.02)
        grads = [torch.empty(n, dtype=torch.bfloat16, device="cuda")
                 for n in wl.numels]
        flag = torch.full((1,), 7, dtype=torch.int32, device="cuda")
        lr, ils = schedule(1)
        for i, g in enumerate(grads):
            g.copy_(wl.grad(i, 1, "cuda"))
        dev.set_lr(lr)
        dev.state.inv_loss_scale.fill_(ils)
        dev.step(grads, found_inf_dev=flag, stream=s)
    s.synchronize()
    host.lr = lr
    assert host.step(grads, ils) == 0
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        dev.step(grads, found_inf_dev=flag, stream=s)
    for t in range(2, 6):
        lr, ils = schedule(t)
        with torch.cuda.stream(s):
            for i, x in enumerate(grads):
                x.copy_(wl.grad(i, t, "cuda"))
            dev.set_lr(lr)
            dev.state.inv_loss_scale.fill_(ils)
            g.replay()
        s.synchronize()
        host.lr = lr
        assert host.step(grads, ils) == 0
        torch.cuda.synchronize()
        assert flag.item() == 0 and dev.state.step.item() == t
        assert host.last_grad_norm > 0.02           # the clip is active
        assert dev.grad_norm_dev.item() == np.float32(host.last_grad_norm)
        _assert_same(host, dev, p_host, p_dev)
