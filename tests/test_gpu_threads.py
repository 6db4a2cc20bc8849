"""Calls from several host threads on several streams: a call that waits for
its stream (a host found_inf or norm read) must not hold up another thread's
call on another stream.  Thread A queues a bounded device sleep (about half
a second) on its stream, then a step that reads found_inf on the host, so A
blocks until its stream drains; meanwhile thread B's cast on its own stream
must return, and both results must still match the oracle."""
import threading
import time

import numpy as np
import pytest
import torch

import oracle
import synth
from harness import GpuState, fresh_states, oracle_cast, oracle_step, set_grads
from parity import check_codes, check_f32_exact, to_np_u8

pytestmark = pytest.mark.gpu

SLEEP_CYCLES = 1_000_000_000   # ~0.5 s at the GB300's 2 GHz SM clock


@pytest.mark.parametrize("entry", ["adamw", "clipped", "fused"])
def test_host_read_does_not_block_other_streams(entry):
    import bit_optimizer_gb300 as bo
    wl = synth.tiny()
    states = fresh_states(wl.weights(), o3=False)
    codes, _, scale = oracle_cast(wl.grads(1), oracle.E4M3)
    set_grads(states, codes, scale)
    gpu = GpuState([s.copy() for s in states])
    ref = [s.copy() for s in states]
    if entry == "clipped":   # a threshold far above the norm: measures only
        assert oracle.adam_step_clipped(ref, wl.lr, wl.beta1, wl.beta2, wl.eps,
                                        wl.wd, 1, wl.inv_loss_scale, 1e9)[0] == 0
    else:
        assert oracle_step(ref, wl, 1) == 0
    sa, sb = torch.cuda.Stream(), torch.cuda.Stream()
    # B's list, run once first so its workspace and tables exist
    srcs = [g.cuda() for g in wl.grads(2)]
    bcodes = [torch.zeros(g.numel(), dtype=torch.uint8, device="cuda") for g in srcs]
    bamax = torch.zeros(len(srcs), device="cuda")
    bscale = torch.zeros(len(srcs), device="cuda")
    bplan = bo.CastPlan(srcs, bcodes, bamax, bscale, "e4m3")
    bplan(stream=sb)
    fused = None
    if entry == "fused":
        fsrcs = [g.cuda() for g in wl.grads(1)]
        famax = torch.zeros(len(fsrcs), device="cuda")
        fused = bo.CastStepPlan(bo.CastPlan(fsrcs, gpu.g, famax, gpu.g_scale, "e4m3"),
                                gpu.plan)
    torch.cuda.synchronize()

    entered, a_done = threading.Event(), threading.Event()
    out = {}

    def thread_a():
        with torch.cuda.stream(sa):
            torch.cuda._sleep(SLEEP_CYCLES)
            entered.set()
            args = (wl.lr, wl.beta1, wl.beta2, wl.eps, wl.wd, 1, wl.inv_loss_scale)
            if entry == "adamw":
                out["found"] = gpu.plan(*args, stream=sa)
            elif entry == "clipped":
                out["found"] = gpu.plan(*args, stream=sa, max_grad_norm=1e9)
            else:
                out["found"] = fused(*args, stream=sa)
            a_done.set()

    ta = threading.Thread(target=thread_a)
    ta.start()
    assert entered.wait(30)
    time.sleep(0.05)                  # A is now inside its blocking read
    t0 = time.perf_counter()
    bplan(stream=sb)
    b_call = time.perf_counter() - t0
    a_still_blocked = not a_done.is_set()
    sb.synchronize()
    ta.join(60)
    assert not ta.is_alive()
    assert a_still_blocked, f"B's call took {b_call:.3f} s and returned after A's"
    assert out["found"] == 0
    # both results are still right
    gpu.compare(ref)
    o_codes, o_amax, o_scale = oracle_cast(wl.grads(2), oracle.E4M3)
    check_f32_exact(bamax.cpu().numpy(), o_amax, "amax")
    check_f32_exact(bscale.cpu().numpy(), o_scale, "scale")
    for i, (c, r) in enumerate(zip(bcodes, o_codes)):
        check_codes(to_np_u8(c), r, oracle.E4M3, name=f"codes[{i}]")
