"""fp8_cast_scaled_noalloc: the cast entry point for callers that must not
allocate device memory (for example a runtime whose pool allocator owns all
device memory, or a service that must not stall on an allocation mid-step).
It keeps its scratch in a fixed array inside the library, so these tests
check, through the C ABI, that it returns what the allocating fp8_cast_scaled
returns on the same inputs, and what the oracle returns, on two calls in a row
with different lists (the array keeps the previous call's contents, which
must not leak into the next result); that it refuses lists beyond its fixed
limits before launching anything; and that it refuses a stream that is
capturing a CUDA graph without breaking that capture.

The test allocates its own buffers with torch; only the entry point under
test is forbidden to allocate.  Kept in a file of its own that is collected
last."""
import ctypes as C

import numpy as np
import pytest
import torch

from harness import oracle_cast
from parity import check_codes, check_f32_exact, to_np_u8

pytestmark = pytest.mark.gpu

E4M3, E5M2 = 0, 1


def make_inputs(seed, sizes, dtypes):
    g = torch.Generator().manual_seed(seed)
    out = []
    for i, (n, dt) in enumerate(zip(sizes, dtypes)):
        x = torch.randn(n, generator=g) * 10.0 ** (-(i % 6))
        out.append(x.to(dt).cuda())
    return out


def items_for(lib, srcs, codes, amax, scale):
    items = (lib.CastItem * len(srcs))()
    for i, (s, c) in enumerate(zip(srcs, codes)):
        it = items[i]
        it.src, it.numel = s.data_ptr(), s.numel()
        it.dtype = {torch.float32: 0, torch.bfloat16: 1, torch.float16: 2}[s.dtype]
        it.codes = c.data_ptr()
        it.amax = amax.data_ptr() + 4 * i
        it.scale = scale.data_ptr() + 4 * i
    return items


def run_noalloc(bo, lib, srcs, fmt):
    n = len(srcs)
    # outputs start as garbage, so a result left from an earlier call or a
    # skipped write cannot pass for a correct one
    codes = [torch.full((s.numel(),), 0xA5, dtype=torch.uint8, device="cuda")
             for s in srcs]
    amax = torch.full((n,), -7.0, device="cuda")
    scale = torch.full((n,), -7.0, device="cuda")
    items = items_for(lib, srcs, codes, amax, scale)
    stream = torch.cuda.current_stream().cuda_stream or None
    rc = bo.load().fp8_cast_scaled_noalloc(items, n, fmt, stream)
    assert rc == 0, bo.load().fp8opt_last_error().decode()
    torch.cuda.synchronize()
    return codes, amax, scale


def test_noalloc_matches_the_allocating_cast_on_two_calls():
    import bit_optimizer_gb300 as bo
    from bit_optimizer_gb300 import _lib
    calls = [
        # a long list with multi-chunk and ragged tensors, E4M3
        (1, [300_001, 4096, 1, 0, 77, 65_536, 32_769, 9] * 3,
         [torch.bfloat16, torch.float32, torch.float16, torch.bfloat16] * 6, E4M3),
        # then a shorter list with other values and the other format
        (2, [70_000, 5, 1024], [torch.float16, torch.bfloat16, torch.float32],
         E5M2),
    ]
    for seed, sizes, dtypes, fmt in calls:
        srcs = make_inputs(seed, sizes, dtypes[:len(sizes)])
        ref_codes, ref_amax, ref_scale = bo.fp8_cast_scaled(srcs, fmt)
        torch.cuda.synchronize()
        codes, amax, scale = run_noalloc(bo, _lib, srcs, fmt)
        n = len(srcs)
        check_f32_exact(amax.cpu().numpy(), ref_amax.cpu().numpy()[:n], "amax")
        check_f32_exact(scale.cpu().numpy(), ref_scale.cpu().numpy()[:n], "scale")
        for i, (c, r) in enumerate(zip(codes, ref_codes)):
            check_codes(to_np_u8(c), to_np_u8(r), fmt, name=f"codes[{i}]")
        # and against the oracle on the same values
        o_codes, o_amax, o_scale = oracle_cast([x.cpu() for x in srcs], fmt)
        check_f32_exact(amax.cpu().numpy(), o_amax, "amax (oracle)")
        check_f32_exact(scale.cpu().numpy(), o_scale, "scale (oracle)")
        for i, (c, r) in enumerate(zip(codes, o_codes)):
            check_codes(to_np_u8(c), r, fmt, name=f"codes[{i}] (oracle)")


def test_noalloc_refuses_lists_beyond_its_limits():
    import bit_optimizer_gb300 as bo
    from bit_optimizer_gb300 import _lib
    L = bo.load()
    amax = torch.full((2000,), -7.0, device="cuda")
    scale = torch.full((2000,), -7.0, device="cuda")
    src = torch.zeros(8, dtype=torch.bfloat16, device="cuda")
    code = torch.zeros(8, dtype=torch.uint8, device="cuda")
    too_many = items_for(_lib, [src] * 1025, [code] * 1025, amax, scale)
    assert L.fp8_cast_scaled_noalloc(too_many, 1025, E4M3, None) == _lib.ERR_LIMIT
    assert "maximum of 1024" in L.fp8opt_last_error().decode()
    # one tensor needing more chunks than the array holds: refused before any
    # pointer is used, so its addresses are placeholders
    big = (_lib.CastItem * 1)()
    big[0].src, big[0].codes = src.data_ptr(), code.data_ptr()
    big[0].numel, big[0].dtype = 65536 * 32768 + 1, 1
    big[0].amax, big[0].scale = amax.data_ptr(), scale.data_ptr()
    assert L.fp8_cast_scaled_noalloc(big, 1, E4M3, None) == _lib.ERR_LIMIT
    assert "chunks" in L.fp8opt_last_error().decode()
    torch.cuda.synchronize()
    assert bool((amax == -7.0).all()) and bool((scale == -7.0).all())


def test_noalloc_refuses_a_capturing_stream():
    """Its tables come from host arrays that the next call refills, so a
    stream that is capturing a CUDA graph is refused with an argument error,
    nothing is enqueued, and the caller's capture stays valid."""
    import bit_optimizer_gb300 as bo
    from bit_optimizer_gb300 import _lib
    L = bo.load()
    src = torch.randn(4096, device="cuda").to(torch.bfloat16)
    code = torch.full((4096,), 0xA5, dtype=torch.uint8, device="cuda")
    amax = torch.full((1,), -7.0, device="cuda")
    scale = torch.full((1,), -7.0, device="cuda")
    items = items_for(_lib, [src], [code], amax, scale)
    x = torch.zeros(16, device="cuda")
    side = torch.cuda.Stream()
    graph = torch.cuda.CUDAGraph()
    torch.cuda.synchronize()
    with torch.cuda.graph(graph, stream=side):
        rc = L.fp8_cast_scaled_noalloc(items, 1, E4M3, side.cuda_stream)
        x.add_(1.0)
    assert rc == _lib.ERR_ARG
    assert "capturing" in L.fp8opt_last_error().decode()
    graph.replay()
    graph.replay()
    torch.cuda.synchronize()
    assert bool((x == 2.0).all())
    assert bool((code == 0xA5).all()) and amax.item() == -7.0 and scale.item() == -7.0
    # uncaptured, the same call runs
    assert L.fp8_cast_scaled_noalloc(items, 1, E4M3, side.cuda_stream) == 0
    side.synchronize()
    _, o_amax, o_scale = oracle_cast([src.cpu()], E4M3)
    check_f32_exact(amax.cpu().numpy(), o_amax, "amax")
    check_f32_exact(scale.cpu().numpy(), o_scale, "scale")
