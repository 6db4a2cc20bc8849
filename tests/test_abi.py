"""The C-ABI library: it builds, loads without a GPU, exports every entry
point include/*.h declares, its records have the layout the header gives, and
argument errors come back as status codes before any CUDA call."""
import ctypes as C
import os
import re
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
INCLUDE = os.path.join(ROOT, "include")


@pytest.fixture(scope="module")
def lib():
    import __graft_entry__
    __graft_entry__.build()
    from bit_optimizer_gb300 import _lib
    return _lib


def declared_entry_points():
    names = []
    for f in sorted(os.listdir(INCLUDE)):
        if f.endswith(".h"):
            text = open(os.path.join(INCLUDE, f)).read()
            names += re.findall(r"^FP8OPT_API\s+[\w\s\*]*?\b(\w+)\s*\(", text, re.M)
    return names


def test_every_declared_symbol_is_exported(lib):
    names = declared_entry_points()
    assert {"fp8_cast_scaled", "fp8_adamw_step"} <= set(names)
    L = lib.load()
    for n in names:
        assert hasattr(L, n), n
    assert set(names) == set(lib.EXPORTS)
    out = subprocess.run(["nm", "-D", "--defined-only", lib.LIB_PATH],
                         capture_output=True, text=True, check=True).stdout
    exported = {l.split()[-1] for l in out.splitlines() if " T " in l}
    assert set(names) <= exported


def test_record_layout_matches_header(lib, tmp_path):
    src = tmp_path / "layout.c"
    src.write_text(r'''
#include <stddef.h>
#include <stdio.h>
#include "fp8opt.h"
#define F(T, m) printf(#T "." #m " %zu\n", offsetof(T, m))
int main(void) {
  printf("cast %zu\nparam %zu\nreduce %zu\n", sizeof(fp8opt_cast_item),
         sizeof(fp8opt_param), sizeof(fp8opt_reduce_item));
  F(fp8opt_cast_item, src); F(fp8opt_cast_item, numel); F(fp8opt_cast_item, dtype);
  F(fp8opt_cast_item, codes); F(fp8opt_cast_item, amax); F(fp8opt_cast_item, scale);
  F(fp8opt_param, numel); F(fp8opt_param, g); F(fp8opt_param, g_scale);
  F(fp8opt_param, g_fmt); F(fp8opt_param, m); F(fp8opt_param, m_scale);
  F(fp8opt_param, v); F(fp8opt_param, w); F(fp8opt_param, w8);
  F(fp8opt_param, w8_scale); F(fp8opt_param, w8_amax); F(fp8opt_param, v_bound);
  F(fp8opt_reduce_item, src); F(fp8opt_reduce_item, numel);
  F(fp8opt_reduce_item, stride); F(fp8opt_reduce_item, src_scale);
  F(fp8opt_reduce_item, codes); F(fp8opt_reduce_item, amax);
  F(fp8opt_reduce_item, scale);
  printf("state %zu\n", sizeof(fp8opt_step_state));
  F(fp8opt_step_state, lr); F(fp8opt_step_state, inv_loss_scale);
  F(fp8opt_step_state, step);
  return 0;
}''')
    exe = tmp_path / "layout"
    subprocess.run(["gcc", "-std=c11", "-I", INCLUDE, str(src), "-o", str(exe)],
                   check=True)
    got = dict(l.rsplit(" ", 1) for l in
               subprocess.run([str(exe)], capture_output=True, text=True,
                              check=True).stdout.splitlines())
    assert int(got["cast"]) == C.sizeof(lib.CastItem)
    assert int(got["param"]) == C.sizeof(lib.Param)
    assert int(got["reduce"]) == C.sizeof(lib.ReduceItem)
    # the 16-byte StepState buffer: float lr, float inv_loss_scale, int64 step
    assert int(got["state"]) == 16
    assert (int(got["fp8opt_step_state.lr"]),
            int(got["fp8opt_step_state.inv_loss_scale"]),
            int(got["fp8opt_step_state.step"])) == (0, 4, 8)
    classes = {"fp8opt_cast_item": lib.CastItem, "fp8opt_param": lib.Param,
               "fp8opt_reduce_item": lib.ReduceItem}
    for key, val in got.items():
        if "." in key and not key.startswith("fp8opt_step_state"):
            t, m = key.split(".")
            cls = classes[t]
            assert getattr(cls, m).offset == int(val), key


def test_argument_errors_need_no_gpu(lib):
    L = lib.load()
    item = (lib.CastItem * 1)()
    assert L.fp8_cast_scaled(item, -1, 0, None) == lib.ERR_ARG
    assert L.fp8_cast_scaled(None, 1, 0, None) == lib.ERR_ARG
    assert L.fp8_cast_scaled(item, 1, 7, None) == lib.ERR_UNSUPPORTED
    item[0].dtype = 9
    assert L.fp8_cast_scaled(item, 1, 0, None) == lib.ERR_UNSUPPORTED
    item[0].dtype = 1
    item[0].numel = 10          # NULL src/codes/amax/scale
    assert L.fp8_cast_scaled(item, 1, 0, None) == lib.ERR_ARG
    assert "item 0" in L.fp8opt_last_error().decode()
    assert L.fp8_cast_scaled(item, 0, 0, None) == lib.OK   # empty list

    p = (lib.Param * 1)()
    f = C.c_int(7)
    args = (1e-3, 0.9, 0.999, 1e-8, 0.0)
    assert L.fp8_adamw_step(p, 1, *args, 0, 1.0, C.byref(f), None, None) == lib.ERR_ARG
    assert L.fp8_adamw_step(p, -1, *args, 1, 1.0, C.byref(f), None, None) == lib.ERR_ARG
    p[0].g_fmt = 3
    assert L.fp8_adamw_step(p, 1, *args, 1, 1.0, None, None, None) == lib.ERR_UNSUPPORTED
    p[0].g_fmt = 0
    dummy = C.c_float(1.0)
    p[0].g_scale = p[0].m_scale = C.addressof(dummy)   # pointers never read
    p[0].w8 = 0x1000                                    # w8 without its scales
    assert L.fp8_adamw_step(p, 1, *args, 1, 1.0, None, None, None) == lib.ERR_ARG
    assert "w8" in L.fp8opt_last_error().decode()
    p[0].w8, p[0].w8_scale, p[0].numel = None, C.addressof(dummy), 4
    p[0].g = p[0].m = p[0].v = p[0].w = 0x1000          # never dereferenced
    assert L.fp8_adamw_step(p, 1, *args, 1, 1.0, None, None, None) == lib.ERR_ARG
    assert "O3" in L.fp8opt_last_error().decode()       # incomplete O3 record
    p[0].numel = 0
    assert L.fp8_adamw_step(p, 0, *args, 1, 1.0, C.byref(f), None, None) == lib.OK
    assert f.value == 0


def test_device_step_argument_errors_need_no_gpu(lib):
    L = lib.load()
    p = (lib.Param * 1)()
    item = (lib.CastItem * 1)()
    state = (C.c_int64 * 2)()                     # 16 bytes, 8-aligned
    hp = (0.9, 0.999, 1e-8, 0.0)
    # state NULL or misaligned
    assert L.fp8_adam_step_dev(p, 0, *hp, 0, None, None, None) == lib.ERR_ARG
    assert "state" in L.fp8opt_last_error().decode()
    assert L.fp8_adam_step_dev(p, 0, *hp, 0, C.addressof(state) + 4, None,
                               None) == lib.ERR_ARG
    # l2 must be 0 or 1
    assert L.fp8_adam_step_dev(p, 0, *hp, 2, C.addressof(state), None,
                               None) == lib.ERR_ARG
    assert "l2" in L.fp8opt_last_error().decode()
    # the records are checked as for fp8_adamw_step
    p[0].g_fmt = 3
    assert L.fp8_adam_step_dev(p, 1, *hp, 0, C.addressof(state), None,
                               None) == lib.ERR_UNSUPPORTED
    p[0].g_fmt = 0
    assert L.fp8_adam_step_dev(p, -1, *hp, 0, C.addressof(state), None,
                               None) == lib.ERR_ARG
    assert L.fp8_cast_adamw_step_dev(item, p, 1, 7, *hp, C.addressof(state),
                                     None, None) == lib.ERR_UNSUPPORTED
    assert L.fp8_cast_adamw_step_dev(item, p, 0, 0, *hp, None, None,
                                     None) == lib.ERR_ARG
    # the clipped form: state, l2 and the threshold are checked first
    assert L.fp8_cast_adam_step_clipped_dev(item, p, 0, 0, *hp, 0, 1.0, None,
                                            None, None, None) == lib.ERR_ARG
    assert L.fp8_cast_adam_step_clipped_dev(item, p, 0, 0, *hp, 2, 1.0,
                                            C.addressof(state), None, None,
                                            None) == lib.ERR_ARG
    assert L.fp8_cast_adam_step_clipped_dev(item, p, 0, 0, *hp, 0, float("nan"),
                                            C.addressof(state), None, None,
                                            None) == lib.ERR_ARG
    # nothing was written to the state
    assert list(state) == [0, 0]


def test_fused_call_checks_that_the_step_takes_the_cast_outputs(lib):
    L = lib.load()
    item = (lib.CastItem * 1)()
    p = (lib.Param * 1)()
    dummy = C.c_float(1.0)
    item[0].dtype, item[0].numel = 1, 4
    item[0].src = item[0].codes = 0x1000
    item[0].amax = item[0].scale = C.addressof(dummy)
    p[0].numel = 4
    p[0].g, p[0].g_scale = 0x1000, C.addressof(dummy)
    p[0].m = p[0].v = p[0].w = 0x2000
    p[0].m_scale = C.addressof(dummy)
    args = (1e-3, 0.9, 0.999, 1e-8, 0.0, 1, 1.0, None, None, None)
    p[0].g = 0x3000                                   # not the cast's codes
    assert L.fp8_cast_adamw_step(item, p, 1, 0, *args) == lib.ERR_ARG
    assert "does not take item 0" in L.fp8opt_last_error().decode()
    p[0].g, p[0].g_fmt = 0x1000, 1                    # other format
    assert L.fp8_cast_adamw_step(item, p, 1, 0, *args) == lib.ERR_ARG
    assert L.fp8_cast_adamw_step(item, p, 0, 0, *args) == lib.OK


def test_reduce_argument_errors_need_no_gpu(lib):
    L = lib.load()
    it = (lib.ReduceItem * 1)()
    dummy = C.c_float(1.0)
    assert L.fp8_reduce_scaled(it, -1, 2, 0, 0, 1.0, None) == lib.ERR_ARG
    assert L.fp8_reduce_scaled(it, 1, 0, 0, 0, 1.0, None) == lib.ERR_ARG
    assert L.fp8_reduce_scaled(it, 1, lib.MAX_SHARDS + 1, 0, 0, 1.0, None) == lib.ERR_ARG
    assert L.fp8_reduce_scaled(it, 1, 2, 0, 3, 1.0, None) == lib.ERR_UNSUPPORTED
    assert L.fp8_reduce_scaled(it, 1, 2, 2, 0, 1.0, None) == lib.ERR_UNSUPPORTED
    it[0].numel, it[0].stride = 100, 100            # NULL buffers
    it[0].amax = it[0].scale = C.addressof(dummy)
    assert L.fp8_reduce_scaled(it, 1, 2, 0, 0, 1.0, None) == lib.ERR_ARG
    it[0].src = it[0].codes = it[0].src_scale = 0x1000   # never dereferenced
    it[0].stride = 99                                # stride below numel
    assert L.fp8_reduce_scaled(it, 1, 2, 0, 0, 1.0, None) == lib.ERR_ARG
    assert "item 0" in L.fp8opt_last_error().decode()
    it[0].stride = 2 ** 62                           # k * stride overflows
    assert L.fp8_reduce_scaled(it, 1, 4, 0, 0, 1.0, None) == lib.ERR_ARG
    assert L.fp8_reduce_scaled(it, 0, 2, 0, 0, 1.0, None) == lib.OK
    it[0].stride = 100
    assert L.fp8_reduce_scaled_norm(it, 1, 2, 0, 0, 1.0, 1.0, None, None,
                                    None) == lib.ERR_ARG   # NULL terms
    assert L.fp8_reduce_scaled_norm(it, 0, 2, 0, 0, 1.0, 1.0, None, None,
                                    None) == lib.OK


def test_norm_and_clip_argument_errors_need_no_gpu(lib):
    L = lib.load()
    p = (lib.Param * 1)()
    norm, found = C.c_double(-1.0), C.c_int(7)
    args = (1e-3, 0.9, 0.999, 1e-8, 0.0, 1, 1.0)
    assert L.fp8_grad_norm(p, -1, 1.0, None, None, None, None) == lib.ERR_ARG
    assert L.fp8_grad_norm(p, 0, 1.0, C.byref(norm), None, C.byref(found), None) == lib.OK
    assert norm.value == 0.0 and found.value == 0
    assert L.fp8_adam_step_clipped(p, 0, *args, 2, 1.0, None, None, None, None,
                                   None) == lib.ERR_ARG          # l2 not 0 or 1
    assert L.fp8_adam_step_clipped(p, 0, *args, 0, float("nan"), None, None,
                                   None, None, None) == lib.ERR_ARG
    p[0].g_fmt = 3
    assert L.fp8_adam_step_clipped(p, 1, *args, 0, 1.0, None, None, None, None,
                                   None) == lib.ERR_UNSUPPORTED
    p[0].g_fmt = 0
    assert L.fp8_adam_step_clipped(p, 0, *args, 1, 1.0, C.byref(norm), None,
                                   C.byref(found), None, None) == lib.OK


def test_fused_clip_argument_errors_need_no_gpu(lib):
    L = lib.load()
    item = (lib.CastItem * 1)()
    p = (lib.Param * 1)()
    args = (1e-3, 0.9, 0.999, 1e-8, 0.0, 1, 1.0)
    tail = (None, None, None, None, None)
    assert L.fp8_cast_adam_step_clipped(item, p, 0, 0, *args, 2, 1.0, *tail) == lib.ERR_ARG
    assert L.fp8_cast_adam_step_clipped(item, p, 0, 0, *args, 0, float("nan"),
                                        *tail) == lib.ERR_ARG
    assert L.fp8_cast_adam_step_clipped(item, p, 0, 7, *args, 0, 1.0, *tail) == \
        lib.ERR_UNSUPPORTED
    norm, found = C.c_double(-1.0), C.c_int(7)
    assert L.fp8_cast_adam_step_clipped(item, p, 0, 0, *args, 1, 1.0, C.byref(norm),
                                        None, C.byref(found), None, None) == lib.OK
    assert norm.value == 0.0 and found.value == 0


def test_strerror_texts(lib):
    assert lib.strerror(0) == "success"
    assert lib.strerror(-1) == "invalid argument"
    assert lib.strerror(-4) == "CUDA error"
    assert lib.strerror(-99) == "unknown status"


def test_binding_refuses_cpu_tensors(lib):
    import torch
    import bit_optimizer_gb300 as bo
    with pytest.raises(TypeError):
        bo.CastPlan([torch.zeros(4)], [torch.zeros(4, dtype=torch.uint8)],
                    torch.zeros(1), torch.zeros(1))


def test_step_state_views_match_the_c_layout(lib):
    """StepState's lr, inv_loss_scale and step are views of one 16-byte
    buffer at the offsets of fp8opt_step_state (checked here on a CPU
    buffer)."""
    import struct
    import torch
    from bit_optimizer_gb300.api import StepState
    st = StepState(lr=3e-4, inv_loss_scale=2.0 ** -16, step=41, device="cpu")
    raw = st.buf.numpy().tobytes()
    assert len(raw) == 16
    lr, ils, step = struct.unpack("<ffq", raw)
    assert lr == struct.unpack("<f", struct.pack("<f", 3e-4))[0]
    assert ils == 2.0 ** -16 and step == 41
    st.step.add_(1)
    st.lr.fill_(1e-3)
    lr, ils, step = struct.unpack("<ffq", st.buf.numpy().tobytes())
    assert step == 42 and lr == struct.unpack("<f", struct.pack("<f", 1e-3))[0]
    assert st.step.dtype == torch.int64 and st.lr.dtype == torch.float32



def test_split_step_and_reduction_argument_errors_need_no_gpu(lib):
    """The calls that split the reduction and the step for tensors cut
    across ranks refuse malformed calls before touching the GPU."""
    L = lib.load()
    it = (lib.ReduceItem * 1)()
    assert L.fp8_reduce_scaled_begin(it, 1, 2, 0, 1.0, None, None) == lib.ERR_ARG
    assert L.fp8_reduce_scaled_begin(it, 0, 2, 0, 1.0, None, None) == lib.OK
    assert L.fp8_reduce_scaled_begin(it, -1, 2, 0, 1.0, 0x1000, None) == lib.ERR_ARG
    assert L.fp8_reduce_scaled_finish(it, 1, 2, 0, 0, 1.0, None, 1.0, None, None,
                                      None) == lib.ERR_ARG        # NULL amax bits
    assert L.fp8_reduce_scaled_finish(it, 0, 2, 0, 0, 1.0, None, 1.0, None, 0x1000,
                                      None) == lib.ERR_ARG        # found, no limbs
    assert L.fp8_reduce_scaled_finish(it, 0, 2, 0, 5, 1.0, None, 1.0, None, None,
                                      None) == lib.ERR_UNSUPPORTED
    assert L.fp8_norm_terms_from_limbs(None, None, -1, 0, 1.0, None, None) == lib.ERR_ARG
    assert L.fp8_norm_terms_from_limbs(None, None, 2, 0, 1.0, None, None) == lib.ERR_ARG
    assert L.fp8_norm_terms_from_limbs(None, None, 0, 3, 1.0, None, None) == \
        lib.ERR_UNSUPPORTED
    assert L.fp8_norm_terms_from_limbs(None, None, 0, 0, 1.0, None, None) == lib.OK
    p = (lib.Param * 1)()
    assert L.fp8_adam_step_copy(p, -1, None, None) == lib.ERR_ARG
    assert L.fp8_adam_step_copy(p, 0, None, None) == lib.OK
    args = (1e-3, 0.9, 0.999, 1e-8, 0.0, 1, 1.0)
    assert L.fp8_adam_step_begin(p, 0, *args, 2, None, None, None, None) == lib.ERR_ARG
    assert L.fp8_adam_step_finish(p, 0, *args, 2, None, None, None, None, None,
                                  None) == lib.ERR_ARG
