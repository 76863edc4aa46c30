"""The allocation-free attention entry point, through the C ABI.

mono_attention_noalloc serves callers that cannot allocate device memory -- code running
while a CUDA graph is being captured (an allocation would break the capture), runtimes
without a device allocator, latency-critical host code that must not take the driver's
allocation lock.  Its scratch (split partials, combine counters, status word) is one fixed
array compiled into the library, shared by every call.

Each case runs a layer step (which inserts the rows' KV records and leaves the step's
query in its arena), then calls the entry point twice in a row on that query and cache.
Both outputs must match the oracle's windowed attention on the same query and cache within
the stage tolerance of the parity tests (one bf16 ulp plus 2e-3 of the rms), and must equal
the layer step's own attention output bit for bit (the same kernel and split count, so any
stale partial or counter left in the shared array by the first call would show in the
second).  The windows span one split (small_r11, full_r48), two (the 192-wide non-causal
draft rows of draft_r6) and three (the 300-key window of wide_r9, which also has a pad row).
This file is collected last, so a stop at the first failure has run every other test first.
"""
import ctypes as C

import numpy as np
import pytest
import torch

import gen
import oracle
from tests.gpu_harness import bf16_ulp_check, f16_to_bf16_bits, to_device
from tests.helpers import np_inputs

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


def _splits(spec):
    width = max(spec["window"] if spec["causal"] else spec["swa_width"], spec["window"])
    return (width + 127) // 128


@pytest.mark.parametrize("name,splits", [("small_r11", 1), ("wide_r9", 3), ("draft_r6", 2),
                                         ("full_r48", 1)])
def test_noalloc_attention_matches_oracle_and_layer_step(name, splits):
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    m, f = _entry()
    oracle.build()
    dev = torch.device("cuda")
    full = gen.WORKLOADS[name]["spec"]["hidden"] >= 4096
    spec, w, st = gen.make_workload(name, weight_device=dev if full else "cpu")
    assert _splits(spec) == splits
    wd, sd = to_device(w, st, dev)
    layer = m.Layer(spec, wd)
    cache = sd["kv_cache"].clone()
    out = torch.empty_like(sd["x"])
    layer.step(sd["x"], out, sd["positions"], sd["row_req"], sd["block_table"], cache)
    torch.cuda.synchronize()
    assert layer.status() == 0
    rows, QW = st["rows"], spec["n_q_heads"] * spec["head_dim"]
    o_step = f16_to_bf16_bits(layer.read("o", rows * QW * 2).view(np.float16).reshape(rows, QW))
    q_bits = layer.read("q", rows * QW * 2).view(np.uint16).reshape(rows, QW)
    q_ptr, _ = layer.buffer("q")

    # the oracle on the same query and the cache after the step's insert
    _, sn = np_inputs({}, st)
    rc, o_want = oracle.attention(spec, sn, q_bits, cache=cache.cpu().numpy())
    assert rc == 0

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
        bf16_ulp_check(got, o_want, f"{name}: noalloc call {call} against the oracle")
        assert np.array_equal(got, o_step), f"{name}: noalloc call {call} differs from the step"
        pad = np.asarray(st["positions"]) < 0
        assert not got[pad].any()
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
