"""Library calls captured into CUDA graphs.  A capture records the call's
kernels with its tables and scalars; replays reuse them, zeroing the
per-tensor slots first, so replays with new input values give the same bytes
as direct calls.  The step's scalars (lr, the bias corrections of `step`,
inv_loss_scale) are part of what a capture fixes."""
import numpy as np
import pytest
import torch

import synth

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def bo():
    import bit_optimizer_gb300 as bo
    return bo


@pytest.fixture
def stream(bo):
    """A stream for capturing; its (frozen) workspace is freed afterwards,
    since torch hands the same streams out again."""
    import gc
    s = torch.cuda.Stream()
    yield s
    gc.collect()                    # the test's graphs are destroyed first
    torch.cuda.synchronize()
    bo.release_stream(s)


def test_cast_graph_replays_match_direct_calls(bo, stream):
    wl = synth.gpt2_cast(n_layer=1, d=128, ffn=512, vocab=3000, ctx=64)
    srcs = [torch.empty(n, dtype=torch.bfloat16, device="cuda") for n in wl.numels]
    n = len(srcs)
    codes = [torch.empty(x, dtype=torch.uint8, device="cuda") for x in wl.numels]
    amax, scale = torch.empty(n, device="cuda"), torch.empty(n, device="cuda")
    s = stream
    plan = bo.CastPlan(srcs, codes, amax, scale, "e4m3")
    with torch.cuda.stream(s):
        for i, x in enumerate(srcs):
            x.copy_(wl.grad(i, 1, "cuda"))
        plan(s)                                   # warm-up on the capture stream
    s.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        plan(s)
    ref_codes = [torch.empty_like(c) for c in codes]
    ra, rs = torch.empty_like(amax), torch.empty_like(scale)
    ref = bo.CastPlan(srcs, ref_codes, ra, rs, "e4m3")
    r = torch.cuda.Stream()              # other lists go on other streams
    with pytest.raises(bo.Fp8OptError):
        ref(s)                           # s's workspace belongs to the graph
    for step in (2, 3, 4):
        with torch.cuda.stream(s):
            for i, x in enumerate(srcs):
                x.copy_(wl.grad(i, step, "cuda") * (10.0 ** (step - 3)))
            g.replay()
        s.synchronize()
        ref(r)
        r.synchronize()
        assert torch.equal(amax, ra) and torch.equal(scale, rs)
        for a, b in zip(codes, ref_codes):
            assert torch.equal(a, b)


def test_reduce_graph_replays_match_direct_calls(bo, stream):
    k, sizes = 4, [40000, 8193, 17]
    shards = [torch.empty((k, x), dtype=torch.uint8, device="cuda") for x in sizes]
    scales = torch.empty((len(sizes), k), device="cuda")
    codes = [torch.empty(x, dtype=torch.uint8, device="cuda") for x in sizes]
    amax, scale = torch.empty(3, device="cuda"), torch.empty(3, device="cuda")
    plan = bo.ReducePlan(shards, scales, codes, amax, scale, "e4m3", "e4m3", 0.25)
    rng = np.random.default_rng(0)

    def fill():
        for sh in shards:
            c = rng.integers(0, 256, tuple(sh.shape), dtype=np.uint8)
            c[(c & 0x7F) == 0x7F] &= 0xF7
            sh.copy_(torch.from_numpy(c))
        scales.copy_(torch.from_numpy(rng.uniform(0.5, 4.0, tuple(scales.shape))
                                      .astype(np.float32)))

    s = stream
    with torch.cuda.stream(s):
        fill()
        plan(s)
    s.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        plan(s)
    rc = [torch.empty_like(c) for c in codes]
    ra, rs = torch.empty_like(amax), torch.empty_like(scale)
    ref = bo.ReducePlan(shards, scales, rc, ra, rs, "e4m3", "e4m3", 0.25)
    r = torch.cuda.Stream()
    for _ in range(3):
        with torch.cuda.stream(s):
            fill()
            g.replay()
            plan(s)                      # the captured list itself: allowed
        s.synchronize()
        ref(r)
        r.synchronize()
        assert torch.equal(amax, ra) and torch.equal(scale, rs)
        for a, b in zip(codes, rc):
            assert torch.equal(a, b)


def test_step_graph_replay_is_the_captured_step(bo, stream):
    """A captured fused cast + step, replayed from a restored state, gives the
    bytes of the same step run directly."""
    wl = synth.o3_1p3b(n_layer=1, d=64, ffn=256, vocab=300, ctx=32)
    s = stream
    with torch.cuda.stream(s):
        params = [w.cuda() for w in wl.weights()]
        opt = bo.Fp8AdamW(params, level="O3", max_grad_norm=0.05)
        grads = [torch.empty(x, dtype=torch.bfloat16, device="cuda") for x in wl.numels]
        for i, x in enumerate(grads):
            x.copy_(wl.grad(i, 1, "cuda"))
        flag = torch.zeros(1, dtype=torch.int32, device="cuda")
        opt.step(grads, found_inf_dev=flag, sync=False, stream=s)   # step 1, warm-up
    s.synchronize()
    snap = opt.state_dict()
    w_snap = [p.clone() for p in params]
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        opt.step(grads, found_inf_dev=flag, sync=False, stream=s)   # step 2
    for i, x in enumerate(grads):
        x.copy_(wl.grad(i, 2, "cuda"))

    def restore():
        opt.load_state_dict(snap)
        for p, w in zip(params, w_snap):
            p.copy_(w)

    with torch.cuda.stream(s):
        restore()
        g.replay()
    s.synchronize()
    got = ([p.clone() for p in params], [t.clone() for t in opt.m],
           [t.clone() for t in opt.w8], opt.w8_scale.clone())
    with torch.cuda.stream(s):
        restore()
        assert opt.step(grads, stream=s) == 0                        # step 2 again
    s.synchronize()
    for a, b in zip(got[0], params):
        assert torch.equal(a, b)
    for a, b in zip(got[1], opt.m):
        assert torch.equal(a, b)
    for a, b in zip(got[2], opt.w8):
        assert torch.equal(a, b)
    assert torch.equal(got[3], opt.w8_scale)
    assert flag.item() == 0


def test_new_list_under_capture_is_refused(bo, stream):
    srcs = [torch.ones(1000, device="cuda")]
    codes = [torch.empty(1000, dtype=torch.uint8, device="cuda")]
    amax, scale = torch.empty(1, device="cuda"), torch.empty(1, device="cuda")
    plan = bo.CastPlan(srcs, codes, amax, scale, "e4m3")
    s = stream
    g = torch.cuda.CUDAGraph()
    with pytest.raises(bo.Fp8OptError):
        with torch.cuda.graph(g, stream=s):
            plan(s)                                   # never run on this stream
