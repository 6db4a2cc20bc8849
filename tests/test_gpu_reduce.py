"""GPU parity of fp8_reduce_scaled (local reduction of FP8 shards) against the
oracle, through the C ABI.  Shards and their scales come from the oracle's own
cast of per-rank gradients, or are random codes and scales."""
import numpy as np
import pytest
import torch

import oracle
import synth
from parity import check_codes, check_f32_exact, to_np_u8

pytestmark = pytest.mark.gpu
E4M3, E5M2 = oracle.E4M3, oracle.E5M2


@pytest.fixture(scope="module")
def bo():
    import bit_optimizer_gb300 as bo
    return bo


def bf16_bits(t):
    return t.contiguous().view(torch.int16).numpy().view(np.uint16)


def oracle_shards(wl, in_fmt, step=1):
    """Per tensor: ([k, numel] uint8 codes, [k] float32 scales), each rank's
    gradient cast by the oracle."""
    out = []
    for i in range(len(wl.shapes)):
        codes, scales = [], []
        for r in range(wl.ranks):
            c, _, s = oracle.cast_scaled(bf16_bits(wl.rank_grad(i, step, r)),
                                         oracle.BF16, in_fmt)
            codes.append(c)
            scales.append(s)
        out.append((np.stack(codes), np.array(scales, np.float32)))
    return out


def random_shards(rng, sizes, k, fmt):
    out = []
    for n in sizes:
        c = rng.integers(0, 256, (k, n), dtype=np.uint8)
        nan = (c & 0x7F) == 0x7F if fmt == E4M3 else (c & 0x7C) == 0x7C
        c[nan] &= 0xF7 if fmt == E4M3 else 0xF3
        s = np.float32(rng.uniform(0.5, 2.0, k) * 2.0 ** rng.integers(-6, 7, k))
        out.append((c, s))
    return out


def gpu_reduce(bo, shards, in_fmt, out_fmt, post, pad=0, in_place=False):
    """Runs the library on copies of the shards; pad > 0 gives each tensor a
    row stride of numel + pad (padding filled with NaN codes)."""
    dev_shards, codes = [], []
    for c, _ in shards:
        k, n = c.shape
        buf = torch.full((k, n + pad), 0x7F, dtype=torch.uint8, device="cuda")
        buf[:, :n] = torch.from_numpy(c).cuda()
        view = buf[:, :n]
        dev_shards.append(view)
        codes.append(view[0] if in_place else
                     torch.empty(n, dtype=torch.uint8, device="cuda"))
    scales = torch.from_numpy(np.stack([s for _, s in shards])).cuda()
    n = len(shards)
    amax = torch.empty(n, device="cuda")
    scale = torch.empty(n, device="cuda")
    bo.fp8_reduce_scaled(dev_shards, scales, in_fmt, out_fmt, post, codes=codes,
                         amax=amax, scale=scale)
    torch.cuda.synchronize()
    return ([to_np_u8(c) for c in codes], amax.cpu().numpy(), scale.cpu().numpy())


def compare(bo, shards, in_fmt, out_fmt, post=1.0, **kw):
    got_codes, got_amax, got_scale = gpu_reduce(bo, shards, in_fmt, out_fmt, post, **kw)
    ref = [oracle.reduce_scaled(c, s, in_fmt, out_fmt, post) for c, s in shards]
    check_f32_exact(got_amax, [r[1] for r in ref], "amax")
    check_f32_exact(got_scale, [r[2] for r in ref], "scale")
    exact = [check_codes(g, r[0], out_fmt, name=f"codes[{i}]")
             for i, (g, r) in enumerate(zip(got_codes, ref))]
    return min(exact) if exact else 1.0


@pytest.mark.parametrize("k", [2, 8])
@pytest.mark.parametrize("in_fmt,out_fmt", [(E4M3, E4M3), (E5M2, E4M3), (E5M2, E5M2)])
def test_gpt_list_cast_shards(bo, k, in_fmt, out_fmt):
    wl = synth.fp8_reduce(ranks=k, n_layer=1, d=128, ffn=512, vocab=3000, ctx=64)
    shards = oracle_shards(wl, in_fmt)
    assert compare(bo, shards, in_fmt, out_fmt, 1.0 / k) == 1.0


@pytest.mark.parametrize("k", [1, 2, 3, 4, 5, 8, 64])
def test_ragged_sizes_many_k(bo, k):
    sizes = [0, 1, 15, 16, 17, 4095, 8191, 8192, 8193, 32767, 32768, 32769, 100003]
    if k == 64:
        sizes = [0, 17, 8193, 40000]
    shards = random_shards(np.random.default_rng(k), sizes, k, E4M3)
    assert compare(bo, shards, E4M3, E4M3, 1.0) == 1.0


@pytest.mark.parametrize("k", [1, 2, 4, 8])
def test_padded_stride_and_unaligned_stride(bo, k):
    shards = random_shards(np.random.default_rng(9), [5000, 40000, 33], k, E5M2)
    # stride numel + 16k: vector path where numel is a multiple of 16
    assert compare(bo, shards, E5M2, E4M3, 0.25, pad=48) == 1.0
    # stride numel + 3: not a multiple of 16, scalar path
    assert compare(bo, shards, E5M2, E4M3, 0.25, pad=3) == 1.0


@pytest.mark.parametrize("k", [1, 2, 8])
@pytest.mark.parametrize("post", [0.0, -0.75, 3e37, 1e-40, float("inf")])
def test_post_factors(bo, k, post):
    """Zero, negative, overflowing, subnormal-making and infinite post
    factors: amax, scale and codes against the oracle, in the passes
    specialised on k = 1, 2 and 8."""
    shards = random_shards(np.random.default_rng(50 + k), [0, 17, 40000, 100003],
                           k, E4M3)
    assert compare(bo, shards, E4M3, E4M3, post) >= 0.999
    assert compare(bo, shards, E4M3, E5M2, post) >= 0.999


def test_in_place_into_the_first_shard(bo):
    shards = random_shards(np.random.default_rng(4), [70000, 8192, 100], 3, E4M3)
    assert compare(bo, shards, E4M3, E4M3, 1.0, in_place=True) == 1.0


def test_non_finite_shards(bo):
    rng = np.random.default_rng(12)
    shards = random_shards(rng, [40000, 40000, 40000, 20000], 2, E5M2)
    shards[0][0][1, 777] = 0x7F           # NaN code
    shards[1][0][0, 9000] = 0x7C          # +inf
    shards[2][0][0, 5] = 0x7C             # +inf + -inf = NaN
    shards[2][0][1, 5] = 0xFC
    assert compare(bo, shards, E5M2, E5M2, 1.0) >= 0.999
    assert compare(bo, shards, E5M2, E4M3, 0.5) >= 0.999


def test_cancelling_shards_give_zero_and_unit_scale(bo):
    rng = np.random.default_rng(2)
    c = random_shards(rng, [30000], 1, E4M3)[0][0][0]
    shards = [(np.stack([c, c ^ 0x80]), np.array([2.0, 2.0], np.float32))]
    codes, amax, scale = gpu_reduce(bo, shards, E4M3, E4M3, 1.0)
    assert amax[0] == 0.0 and scale[0] == 1.0 and not codes[0].any()


def test_repeated_calls_on_cached_tables(bo):
    """One plan over fixed buffers, new shard contents each call."""
    k, sizes = 4, [50000, 300]
    dev = [torch.empty((k, n), dtype=torch.uint8, device="cuda") for n in sizes]
    sc = torch.empty((2, k), device="cuda")
    codes = [torch.empty(n, dtype=torch.uint8, device="cuda") for n in sizes]
    amax, scale = torch.empty(2, device="cuda"), torch.empty(2, device="cuda")
    plan = bo.ReducePlan(dev, sc, codes, amax, scale, "e4m3", "e4m3", 0.25)
    rng = np.random.default_rng(21)
    for call in range(3):
        shards = random_shards(rng, sizes, k, E4M3)
        for d, (c, _) in zip(dev, shards):
            d.copy_(torch.from_numpy(c))
        sc.copy_(torch.from_numpy(np.stack([s for _, s in shards])))
        plan()
        torch.cuda.synchronize()
        for i, (c, s) in enumerate(shards):
            rc, ra, rs = oracle.reduce_scaled(c, s, E4M3, E4M3, 0.25)
            check_f32_exact(amax.cpu().numpy()[i:i + 1], [ra], f"amax {call}")
            check_f32_exact(scale.cpu().numpy()[i:i + 1], [rs], f"scale {call}")
            assert np.array_equal(to_np_u8(codes[i]), rc)



@pytest.mark.parametrize("k", [1, 2, 3, 4, 8])
@pytest.mark.parametrize("out_fmt", [E4M3, E5M2])
def test_reduce_with_norm_terms(bo, out_fmt, k):
    """fp8_reduce_scaled_norm: the outputs of fp8_reduce_scaled plus each
    tensor's norm term of its output codes, bit-exact against the oracle's
    terms of the oracle's reduction (k = 1, 2, 4, 8 take the encode pass
    specialised on k; the 100003-element tensor has whole 32768-element
    chunks and a ragged end)."""
    sizes = [0, 17, 8193, 40000, 100003, 98304]
    shards = random_shards(np.random.default_rng(31 + out_fmt + 10 * k), sizes,
                           k, E4M3)
    ils = 2.0 ** -3
    dev = [torch.from_numpy(c).cuda() for c, _ in shards]
    scales = torch.from_numpy(np.stack([s for _, s in shards])).cuda()
    codes = [torch.empty(c.shape[1], dtype=torch.uint8, device="cuda") for c, _ in shards]
    n_t = len(sizes)
    amax, scale = torch.empty(n_t, device="cuda"), torch.empty(n_t, device="cuda")
    terms = torch.full((n_t,), -1.0, dtype=torch.float64, device="cuda")
    found = torch.full((1,), 7, dtype=torch.int32, device="cuda")
    plan = bo.ReducePlan(dev, scales, codes, amax, scale, "e4m3",
                         {E4M3: "e4m3", E5M2: "e5m2"}[out_fmt], 1.0 / k)
    plan(norm_terms=terms, found=found, inv_loss_scale=ils)
    torch.cuda.synchronize()
    ref = [oracle.reduce_scaled(c, s, E4M3, out_fmt, 1.0 / k) for c, s in shards]
    states = [oracle.StepState(rc, float(rs), np.zeros(rc.size, np.uint8), 1.0,
                               np.zeros(rc.size, np.uint16), np.zeros(rc.size, np.uint16),
                               g_fmt=out_fmt) for rc, _, rs in ref]
    f, tt = oracle.grad_norm_terms(states, ils)
    assert found.item() == f == 0
    assert np.array_equal(terms.cpu().numpy(), tt)
    for c, (rc, ra, rs) in zip(codes, ref):
        assert np.array_equal(to_np_u8(c), rc)
    # finite codes whose values overflow once unscaled: found_inf from the
    # overflow threshold, as the oracle decides it
    big = 2.0 ** 120
    plan(norm_terms=terms, found=found, inv_loss_scale=big)
    torch.cuda.synchronize()
    f_big, _ = oracle.grad_norm_terms(states, big)
    assert found.item() == f_big == 1
    # a NaN code in a shard: found_inf
    shards[3][0][k - 1, 5] = 0x7F
    dev[3].copy_(torch.from_numpy(shards[3][0]))
    plan(norm_terms=terms, found=found, inv_loss_scale=ils)
    torch.cuda.synchronize()
    assert found.item() == 1
