"""The C-ABI library loads, exports every function include/mono_layer.h declares, and the
binding's structures have the header's layout.  No GPU needed: nothing computes."""
import ctypes as C
import os
import re
import subprocess
import sys

import pytest

import moe_decode_layer_mxfp8_gb300 as m

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "mono_layer.h")


@pytest.fixture(scope="module")
def built():
    from moe_decode_layer_mxfp8_gb300 import build
    build.build()
    return m.lib()


def _declared():
    text = open(HEADER).read()
    return sorted(set(re.findall(r"\b(mono_\w+)\s*\(", text)))


def test_every_declared_function_is_exported(built):
    names = _declared()
    assert set(names) == set(m.EXPORTS), (names, m.EXPORTS)
    out = subprocess.run(["nm", "-D", "--defined-only", m.LIB_PATH], capture_output=True, text=True).stdout
    exported = set(re.findall(r"\bT (mono_\w+)", out))
    assert set(names) <= exported, set(names) - exported
    for n in names:
        assert hasattr(built, n)


def test_strerror_without_gpu(built):
    assert m.strerror(0) == "ok"
    assert "rows" in m.strerror(-3)
    assert m.strerror(12345) == "unknown error"


def test_null_arguments_are_refused(built):
    h = C.c_void_p()
    assert built.mono_layer_build(None, None, C.byref(h)) == -1
    assert built.mono_layer_step(None, None, None) == -1
    assert built.mono_ffn_step(None, None, None) == -1
    assert built.mono_layer_selftest_wait_timeout(None, 1000000, None) == -1
    assert built.mono_layer_status(None, 0) == -1
    built.mono_layer_free(None)


def test_bad_spec_is_refused_before_touching_the_device(built):
    import gen
    spec = gen.spec_of("tiny", max_rows=1)
    w = m.Weights(**{k: 16 * (i + 1) for i, k in enumerate(m.WEIGHT_FIELDS)})
    h = C.c_void_p()
    bad = dict(spec, hidden=250)
    assert built.mono_layer_build(C.byref(m.make_spec(bad)), C.byref(w), C.byref(h)) == -2
    bad = dict(spec, max_rows=49)
    assert built.mono_layer_build(C.byref(m.make_spec(bad)), C.byref(w), C.byref(h)) == -3
    bad = dict(spec, head_dim=96)
    assert built.mono_layer_build(C.byref(m.make_spec(bad)), C.byref(w), C.byref(h)) == -2
    w2 = m.Weights(**{k: 16 * (i + 1) + (3 if k == "wq_b" else 0) for i, k in enumerate(m.WEIGHT_FIELDS)})
    assert built.mono_layer_build(C.byref(m.make_spec(spec)), C.byref(w2), C.byref(h)) == -4


def test_struct_layout_matches_header(tmp_path):
    src = tmp_path / "layout.c"
    src.write_text("""
#include <stdio.h>
#include <stddef.h>
#include "mono_layer.h"
int main(void) {
  printf("%zu %zu %zu\\n", sizeof(mono_layer_spec), sizeof(mono_layer_weights), sizeof(mono_step_args));
  printf("%zu %zu %zu %zu\\n", offsetof(mono_layer_spec, eps), offsetof(mono_step_args, rows),
         offsetof(mono_step_args, kv_cache), offsetof(mono_step_args, topk_w_out));
  printf("%zu %zu %zu\\n", sizeof(mono_ffn_args), offsetof(mono_ffn_args, rows),
         offsetof(mono_ffn_args, topk_w_out));
  return 0;
}
""")
    exe = tmp_path / "layout"
    subprocess.run(["gcc", "-I", os.path.join(ROOT, "include"), str(src), "-o", str(exe)], check=True)
    got = subprocess.run([str(exe)], capture_output=True, text=True, check=True).stdout.split()
    want = [C.sizeof(m.Spec), C.sizeof(m.Weights), C.sizeof(m.StepArgs), m.Spec.eps.offset,
            m.StepArgs.rows.offset, m.StepArgs.kv_cache.offset, m.StepArgs.topk_w_out.offset,
            C.sizeof(m.FfnArgs), m.FfnArgs.rows.offset, m.FfnArgs.topk_w_out.offset]
    assert [int(v) for v in got] == want


def test_attention_weights_all_or_none(built):
    import gen
    spec = gen.spec_of("tiny", max_rows=1)
    h = C.c_void_p()
    half = {k: (None if k in ("wqkv", "wo_b_s") else 16 * (i + 1)) for i, k in enumerate(m.WEIGHT_FIELDS)}
    assert built.mono_layer_build(C.byref(m.make_spec(spec)), C.byref(m.Weights(**half)), C.byref(h)) == -1
    ffn = {k: (None if k in m.ATTN_WEIGHT_FIELDS else 16 * (i + 1)) for i, k in enumerate(m.WEIGHT_FIELDS)}
    # an FFN-only handle still checks the FFN fields
    bad = dict(spec, moe_inter=100)
    assert built.mono_layer_build(C.byref(m.make_spec(bad)), C.byref(m.Weights(**ffn)), C.byref(h)) == -2
    ffn["router"] = None
    assert built.mono_layer_build(C.byref(m.make_spec(spec)), C.byref(m.Weights(**ffn)), C.byref(h)) == -1


def test_missing_library_fails_loudly(tmp_path):
    """No fallback: without libmono_layer.so the binding raises instead of computing anything."""
    code = f"""
import sys
sys.path.insert(0, {ROOT!r})
import moe_decode_layer_mxfp8_gb300 as m
m.LIB_PATH = {str(tmp_path / 'absent.so')!r}
try:
    m.lib()
except RuntimeError as e:
    assert 'no CPU fallback' in str(e)
    print('raised')
"""
    out = subprocess.run([sys.executable, "-c", code], capture_output=True, text=True)
    assert out.stdout.strip() == "raised", out.stderr


def test_noalloc_attention_refuses_misaligned_pointers_before_touching_the_device(built):
    """mono_attention_noalloc reads q and writes o in 16-byte vectors: an unaligned q, o or
    cache base is refused with MONO_ERR_BAD_ALIGNMENT on the host (these fake addresses are
    never dereferenced, and no device is needed)."""
    import gen
    f = built.mono_attention_noalloc
    f.restype = C.c_int
    f.argtypes = [C.POINTER(m.Spec), C.c_void_p, C.c_void_p, C.c_void_p, C.c_void_p, C.c_void_p,
                  C.c_int32, C.c_int32, C.c_int32, C.c_void_p, C.c_int64, C.c_int64, C.c_int64,
                  C.c_void_p]
    sp = m.make_spec(gen.spec_of("full_r48", max_rows=48))
    ok, cache = 0x10000, 0x20000

    def call(q, o, kv):
        return f(C.byref(sp), q, o, ok, ok, ok, 4, 1, 8, kv, 128 * 528, 528, 4, None)

    assert call(ok + 2, ok, cache) == -4     # q
    assert call(ok, ok + 8, cache) == -4     # o
    assert call(ok, ok, cache + 4) == -4     # cache base
    assert f(C.byref(sp), ok, ok, ok, ok, ok, 4, 1, 8, cache, 128 * 528, 520, 4, None) == -4  # stride
    assert f(C.byref(sp), ok, ok, ok, ok, ok, 4, 1, 8, cache, 128 * 528 - 16, 528, 4, None) == -5
