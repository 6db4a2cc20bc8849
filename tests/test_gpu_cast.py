"""GPU parity of fp8_cast_scaled against the oracle, through the C ABI."""
import numpy as np
import pytest
import torch

import oracle
import synth
from harness import oracle_cast
from parity import check_codes, check_f32_exact, to_np_u8

pytestmark = pytest.mark.gpu
E4M3, E5M2 = oracle.E4M3, oracle.E5M2


@pytest.fixture(scope="module")
def bo():
    import bit_optimizer_gb300 as bo
    return bo


def gpu_cast(bo, srcs, fmt):
    codes, amax, scale = bo.fp8_cast_scaled(srcs, fmt)
    torch.cuda.synchronize()
    n = len(srcs)
    return ([to_np_u8(c) for c in codes], amax.cpu().numpy()[:n],
            scale.cpu().numpy()[:n])


def compare(bo, host_grads, dev_grads, fmt):
    ref_codes, ref_amax, ref_scale = oracle_cast(host_grads, fmt)
    codes, amax, scale = gpu_cast(bo, dev_grads, fmt)
    check_f32_exact(amax, ref_amax, "amax")
    check_f32_exact(scale, ref_scale, "scale")
    exact = [check_codes(c, r, fmt, name=f"codes[{i}]")
             for i, (c, r) in enumerate(zip(codes, ref_codes))]
    return min(exact) if exact else 1.0


@pytest.mark.parametrize("fmt", [E4M3, E5M2])
def test_gpt_shaped_list_reduced(bo, fmt):
    wl = synth.gpt2_cast(n_layer=2, d=128, ffn=512, vocab=3000, ctx=64)
    grads = wl.grads(step=1)
    assert compare(bo, grads, [g.cuda() for g in grads], fmt) == 1.0


@pytest.mark.parametrize("fmt", [E4M3, E5M2])
@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16, torch.float16])
def test_ragged_sizes_every_dtype(bo, fmt, dtype):
    sizes = [0, 1, 7, 8, 9, 15, 4095, 4096, 4097, 8191, 32767, 32768, 32769,
             65543, 100003]
    g = torch.Generator().manual_seed(17)
    grads = [(torch.randn(n, generator=g) * 10.0 ** (-(i % 7))).to(dtype)
             for i, n in enumerate(sizes)]
    assert compare(bo, grads, [x.cuda() for x in grads], fmt) == 1.0


@pytest.mark.parametrize("fmt", [E4M3, E5M2])
def test_edge_values(bo, fmt):
    inf, nan = float("inf"), float("nan")
    cases = [
        torch.zeros(5000),                                    # all zero
        torch.tensor([1.0, -2.0, inf, 0.5] * 3000),           # +inf
        torch.tensor([-inf, 3.0] * 5000),                     # -inf
        torch.tensor([1.0, nan, -5.0] * 3000),                # NaN
        torch.tensor([1e-45, -1e-45] * 20),                   # scale overflow
        torch.tensor([3.4e38, -1.0, 1e-30] * 4000),           # huge amax
        torch.tensor([-0.0, 0.0, -1e-40, 2e-38] * 4000),      # zeros, subnormals
        torch.tensor([448.0, 464.0, -57344.0, 61440.0] * 10), # near the maxima
    ]
    assert compare(bo, cases, [c.cuda() for c in cases], fmt) == 1.0


def test_unaligned_buffers_take_the_scalar_path(bo):
    g = torch.Generator().manual_seed(3)
    host = [torch.randn(n, generator=g).to(torch.bfloat16) for n in (40001, 4096, 77)]
    dev = []
    for h in host:
        buf = torch.zeros(h.numel() + 1, dtype=h.dtype, device="cuda")
        buf[1:] = h.cuda()
        dev.append(buf[1:])          # 2-byte offset: not 16-byte aligned
    assert dev[0].data_ptr() % 16 != 0
    ref_codes, ref_amax, ref_scale = oracle_cast(host, E4M3)
    outs = []
    for h in host:
        b = torch.zeros(h.numel() + 1, dtype=torch.uint8, device="cuda")
        outs.append(b[1:])
    amax = torch.empty(3, device="cuda")
    scale = torch.empty(3, device="cuda")
    bo.fp8_cast_scaled(dev, E4M3, codes=outs, amax=amax, scale=scale)
    torch.cuda.synchronize()
    check_f32_exact(amax.cpu().numpy(), ref_amax)
    check_f32_exact(scale.cpu().numpy(), ref_scale)
    for o, r in zip(outs, ref_codes):
        assert np.array_equal(to_np_u8(o), r)


def test_repeated_calls_on_cached_tables(bo):
    """The same buffers with new contents: the cached tables must not hold
    stale amax or scale (per-call epochs)."""
    srcs = [torch.empty(70000, dtype=torch.bfloat16, device="cuda"),
            torch.empty(300, dtype=torch.bfloat16, device="cuda")]
    codes = [torch.empty(s.numel(), dtype=torch.uint8, device="cuda") for s in srcs]
    amax = torch.empty(2, device="cuda")
    scale = torch.empty(2, device="cuda")
    plan = bo.CastPlan(srcs, codes, amax, scale, "e4m3")
    g = torch.Generator().manual_seed(5)
    for k, mag in enumerate((1e-3, 5.0, 1e-6, 0.0)):
        host = [(torch.randn(s.numel(), generator=g) * mag).to(torch.bfloat16)
                for s in srcs]
        for s, h in zip(srcs, host):
            s.copy_(h)
        plan()
        torch.cuda.synchronize()
        ref_codes, ref_amax, ref_scale = oracle_cast(host, E4M3)
        check_f32_exact(amax.cpu().numpy(), ref_amax, f"amax call {k}")
        check_f32_exact(scale.cpu().numpy(), ref_scale, f"scale call {k}")
        for c, r in zip(codes, ref_codes):
            assert np.array_equal(to_np_u8(c), r)


def test_status_codes_through_the_binding(bo):
    with pytest.raises(bo.Fp8OptError) as e:
        item = (bo._lib.CastItem * 1)()
        bo._lib.check(bo.load().fp8_cast_scaled(item, 1, 5, None))
    assert e.value.status == -2
