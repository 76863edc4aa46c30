"""The allocation-free attention entry point against the layer step's own attention.

mono_attention_noalloc serves callers that cannot allocate device memory (code running
under CUDA-graph capture, runtimes without a device allocator): its scratch is a fixed
array inside the library.  Here it is called twice in a row through the C ABI on the query
and KV cache a layer step just used; both outputs must match the step's attention output
within the tolerance of the stage parity tests (one bf16 ulp).  The second call shows that
the shared scratch is cleared between calls.
"""
import ctypes as C

import numpy as np
import pytest
import torch

import gen
from tests.gpu_harness import bf16_ulp_check, f16_to_bf16_bits, to_device

pytestmark = pytest.mark.gpu


def _entry():
    import moe_decode_layer_mxfp8_gb300 as m
    from moe_decode_layer_mxfp8_gb300 import build
    build.build()
    L = m.lib()
    f = L.mono_attention_noalloc
    f.restype = C.c_int
    f.argtypes = [C.POINTER(m.Spec), C.c_void_p, C.c_void_p, C.c_void_p, C.c_void_p, C.c_void_p,
                  C.c_int32, C.c_int32, C.c_int32, C.c_void_p, C.c_int64, C.c_int64, C.c_int64,
                  C.c_void_p]
    return m, f


@pytest.mark.parametrize("name", ["small_r11", "full_r48"])
def test_noalloc_attention_matches_layer_step(name):
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    m, f = _entry()
    dev = torch.device("cuda")
    full = gen.WORKLOADS[name]["spec"]["hidden"] >= 4096
    spec, w, st = gen.make_workload(name, weight_device=dev if full else "cpu")
    wd, sd = to_device(w, st, dev)
    layer = m.Layer(spec, wd)
    cache = sd["kv_cache"].clone()
    out = torch.empty_like(sd["x"])
    layer.step(sd["x"], out, sd["positions"], sd["row_req"], sd["block_table"], cache)
    torch.cuda.synchronize()
    assert layer.status() == 0
    rows, QW = st["rows"], spec["n_q_heads"] * spec["head_dim"]
    o_step = f16_to_bf16_bits(layer.read("o", rows * QW * 2).view(np.float16).reshape(rows, QW))
    q_ptr, _ = layer.buffer("q")

    stream = torch.cuda.current_stream()
    sp = m.make_spec(spec)
    for call in range(2):
        o = torch.full((rows, QW), float("nan"), dtype=torch.float16, device=dev)
        rc = f(C.byref(sp), q_ptr, o.data_ptr(), sd["positions"].data_ptr(),
               sd["row_req"].data_ptr(), sd["block_table"].data_ptr(), sd["block_table"].shape[1],
               sd["block_table"].shape[0], rows, cache.data_ptr(), cache.stride(0),
               cache.stride(1), cache.shape[0], C.c_void_p(stream.cuda_stream))
        assert rc == 0, m.strerror(rc)
        torch.cuda.synchronize()
        got = f16_to_bf16_bits(o.cpu().numpy())
        bf16_ulp_check(got, o_step, f"noalloc call {call}")
    layer.close()


def test_noalloc_refuses_too_many_rows():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    m, f = _entry()
    sp = m.make_spec(gen.spec_of("full_r48", max_rows=48))
    d = torch.zeros(16, dtype=torch.int32, device="cuda")
    cache = torch.zeros((4, 128, 528), dtype=torch.uint8, device="cuda")
    rc = f(C.byref(sp), d.data_ptr(), d.data_ptr(), d.data_ptr(), d.data_ptr(), d.data_ptr(), 1, 1,
           49, cache.data_ptr(), cache.stride(0), cache.stride(1), 4, None)
    assert rc == -3
