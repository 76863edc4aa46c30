"""Python binding of the fused MoE decode layer's C ABI (include/mono_layer.h).

Argument marshalling only: every step of the layer runs in the library's CUDA kernels.
PyTorch supplies device memory and the current stream.  Importing works without a GPU;
building or stepping a layer needs libmono_layer.so (``moe_decode_layer_mxfp8_gb300.build``)
and an sm_103 device, and raises if either is missing -- there is no fallback.
"""
from __future__ import annotations

import ctypes as C
import os

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libmono_layer.so")

MONO_OK = 0
ERRORS = {
    -1: "MONO_ERR_INVALID_ARG", -2: "MONO_ERR_UNSUPPORTED_DIMS", -3: "MONO_ERR_TOO_MANY_ROWS",
    -4: "MONO_ERR_BAD_ALIGNMENT", -5: "MONO_ERR_BAD_KV_VIEW", -6: "MONO_ERR_UNSUPPORTED_DEVICE",
    -7: "MONO_ERR_CUDA", -8: "MONO_ERR_OUT_OF_MEMORY", -9: "MONO_ERR_DEVICE_STATUS",
}
STATUS_UNMAPPED_PAGE, STATUS_WAIT_TIMEOUT, STATUS_BAD_ROUTE, STATUS_F16_RANGE = 1, 2, 4, 8

BUF = dict(xn=0, qkv=1, qlatn=2, kvn=3, q=4, o=5, oa=6, h=7, u=8, logits=9, topk_idx=10,
           topk_w=11, slot_pos=12, ts=13, ys=14, tr=15, yr=16)

SPEC_INT_FIELDS = ["hidden", "n_q_heads", "head_dim", "kv_dim", "q_rank", "o_rank", "n_experts",
                   "topk", "moe_inter", "shared_inter", "window", "swa_width", "causal",
                   "block_size", "kv_record_bytes", "max_rows"]
SPEC_FLOAT_FIELDS = ["eps", "swiglu_clamp", "routed_scale"]
ATTN_WEIGHT_FIELDS = ["attn_norm", "q_norm", "kv_norm", "wqkv", "wqkv_s", "wq_b", "wq_b_s", "wo_a",
                      "wo_a_s", "wo_b", "wo_b_s"]
WEIGHT_FIELDS = ["attn_norm", "q_norm", "kv_norm", "ffn_norm", "wqkv", "wqkv_s", "wq_b", "wq_b_s",
                 "wo_a", "wo_a_s", "wo_b", "wo_b_s", "router", "sh_gu", "sh_gu_s", "sh_d", "sh_d_s",
                 "ex_gu", "ex_gu_s", "ex_d", "ex_d_s"]


class Spec(C.Structure):
    _fields_ = [(n, C.c_int32) for n in SPEC_INT_FIELDS] + [(n, C.c_float) for n in SPEC_FLOAT_FIELDS]


class Weights(C.Structure):
    _fields_ = [(n, C.c_void_p) for n in WEIGHT_FIELDS]


class StepArgs(C.Structure):
    _fields_ = [("x_in", C.c_void_p), ("x_out", C.c_void_p), ("positions", C.c_void_p),
                ("row_req", C.c_void_p), ("block_table", C.c_void_p), ("max_blocks", C.c_int32),
                ("n_req", C.c_int32), ("rows", C.c_int32), ("kv_cache", C.c_void_p),
                ("kv_stride_block", C.c_int64), ("kv_stride_tok", C.c_int64),
                ("kv_num_blocks", C.c_int64), ("topk_idx_out", C.c_void_p),
                ("topk_w_out", C.c_void_p)]


class FfnArgs(C.Structure):
    _fields_ = [("x_in", C.c_void_p), ("attn_in", C.c_void_p), ("x_out", C.c_void_p),
                ("positions", C.c_void_p), ("rows", C.c_int32), ("topk_idx_out", C.c_void_p),
                ("topk_w_out", C.c_void_p)]


EXPORTS = ["mono_layer_build", "mono_layer_step", "mono_ffn_step", "mono_layer_status",
           "mono_layer_free",
           "mono_layer_strerror", "mono_layer_buffer", "mono_layer_read_buffer",
           "mono_layer_launches_per_step", "mono_layer_kernels_last_step",
           "mono_layer_launch_name",
           "mono_layer_set_profile_events", "mono_attention_noalloc",
           "mono_layer_selftest_wait_timeout"]

_lib = None


class MonoError(RuntimeError):
    def __init__(self, code: int, what: str):
        super().__init__(f"{what}: {ERRORS.get(code, code)} ({strerror(code)})")
        self.code = code


def lib() -> C.CDLL:
    """The loaded C library; raises if it has not been built."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"{LIB_PATH} is missing: run `python -m moe_decode_layer_mxfp8_gb300.build`"
                               " (the layer has no CPU fallback)")
        L = C.CDLL(LIB_PATH)
        L.mono_layer_build.argtypes = [C.POINTER(Spec), C.POINTER(Weights), C.POINTER(C.c_void_p)]
        L.mono_layer_step.argtypes = [C.c_void_p, C.POINTER(StepArgs), C.c_void_p]
        L.mono_ffn_step.argtypes = [C.c_void_p, C.POINTER(FfnArgs), C.c_void_p]
        L.mono_layer_status.argtypes = [C.c_void_p, C.c_int]
        L.mono_layer_free.argtypes = [C.c_void_p]
        L.mono_layer_free.restype = None
        L.mono_layer_strerror.argtypes = [C.c_int]
        L.mono_layer_strerror.restype = C.c_char_p
        L.mono_layer_buffer.argtypes = [C.c_void_p, C.c_int, C.POINTER(C.c_void_p),
                                        C.POINTER(C.c_size_t)]
        L.mono_layer_read_buffer.argtypes = [C.c_void_p, C.c_int, C.c_void_p, C.c_size_t]
        L.mono_layer_launches_per_step.argtypes = [C.c_void_p]
        L.mono_layer_kernels_last_step.argtypes = [C.c_void_p]
        L.mono_layer_launch_name.argtypes = [C.c_int]
        L.mono_layer_launch_name.restype = C.c_char_p
        L.mono_layer_set_profile_events.argtypes = [C.c_void_p, C.c_void_p, C.c_int]
        L.mono_layer_selftest_wait_timeout.argtypes = [C.c_void_p, C.c_int64, C.c_void_p]
        _lib = L
    return _lib


def strerror(code: int) -> str:
    return lib().mono_layer_strerror(code).decode()


def _ptr(t) -> int | None:
    if t is None:
        return None
    return t.data_ptr()


def make_spec(spec: dict, max_rows: int | None = None) -> Spec:
    d = dict(spec)
    if max_rows is not None:
        d["max_rows"] = max_rows
    return Spec(**{k: d[k] for k in SPEC_INT_FIELDS + SPEC_FLOAT_FIELDS})


class Layer:
    """A built layer: owns the C handle.  ``weights`` maps field names to CUDA tensors that
    must outlive the Layer (they are read in place).  Without any of the attention weights
    the handle is FFN-only and runs ``ffn_step`` alone."""

    def __init__(self, spec: dict, weights: dict, max_rows: int | None = None):
        self.spec = dict(spec)
        self._weights = {k: weights.get(k) for k in WEIGHT_FIELDS}  # keep alive
        self._h = C.c_void_p()
        w = Weights(**{k: _ptr(v) for k, v in self._weights.items()})
        rc = lib().mono_layer_build(C.byref(make_spec(spec, max_rows)), C.byref(w), C.byref(self._h))
        if rc != MONO_OK:
            raise MonoError(rc, "mono_layer_build")
        self.max_rows = max_rows if max_rows is not None else spec["max_rows"]

    def step_args(self, x_in, x_out, positions, row_req, block_table, kv_cache,
                  topk_idx_out=None, topk_w_out=None) -> StepArgs:
        assert kv_cache.dim() == 3, "kv_cache is a [blocks, block_size, record] byte view"
        es = kv_cache.element_size()
        return StepArgs(x_in=_ptr(x_in), x_out=_ptr(x_out), positions=_ptr(positions),
                        row_req=_ptr(row_req), block_table=_ptr(block_table),
                        max_blocks=block_table.shape[1], n_req=block_table.shape[0],
                        rows=x_in.shape[0], kv_cache=_ptr(kv_cache),
                        kv_stride_block=kv_cache.stride(0) * es, kv_stride_tok=kv_cache.stride(1) * es,
                        kv_num_blocks=kv_cache.shape[0], topk_idx_out=_ptr(topk_idx_out),
                        topk_w_out=_ptr(topk_w_out))

    def step(self, x_in, x_out, positions, row_req, block_table, kv_cache, stream=None,
             topk_idx_out=None, topk_w_out=None) -> None:
        """Enqueues one layer step on `stream` (default: torch's current stream)."""
        import torch
        if stream is None:
            stream = torch.cuda.current_stream()
        a = self.step_args(x_in, x_out, positions, row_req, block_table, kv_cache, topk_idx_out,
                           topk_w_out)
        self.step_raw(a, stream.cuda_stream)

    def step_raw(self, args: StepArgs, stream_handle: int) -> None:
        rc = lib().mono_layer_step(self._h, C.byref(args), C.c_void_p(stream_handle))
        if rc != MONO_OK:
            raise MonoError(rc, "mono_layer_step")

    def ffn_step(self, x_in, attn_in, x_out, positions, stream=None, topk_idx_out=None,
                 topk_w_out=None) -> None:
        """Enqueues one FFN launch (residual x_in + attn_in, then the FFN seam and the MoE)
        on `stream` (default: torch's current stream)."""
        import torch
        if stream is None:
            stream = torch.cuda.current_stream()
        a = FfnArgs(x_in=_ptr(x_in), attn_in=_ptr(attn_in), x_out=_ptr(x_out),
                    positions=_ptr(positions), rows=x_in.shape[0], topk_idx_out=_ptr(topk_idx_out),
                    topk_w_out=_ptr(topk_w_out))
        self.ffn_step_raw(a, stream.cuda_stream)

    def ffn_step_raw(self, args: FfnArgs, stream_handle: int) -> None:
        rc = lib().mono_ffn_step(self._h, C.byref(args), C.c_void_p(stream_handle))
        if rc != MONO_OK:
            raise MonoError(rc, "mono_ffn_step")

    def selftest_wait_timeout(self, budget_ns: int, stream=None) -> None:
        """Enqueues a bounded wait that runs out (the status word's WAIT_TIMEOUT bit)."""
        import torch
        if stream is None:
            stream = torch.cuda.current_stream()
        rc = lib().mono_layer_selftest_wait_timeout(self._h, int(budget_ns), C.c_void_p(stream.cuda_stream))
        if rc != MONO_OK:
            raise MonoError(rc, "mono_layer_selftest_wait_timeout")

    def status(self, clear: bool = False) -> int:
        rc = lib().mono_layer_status(self._h, int(clear))
        if rc < 0:
            raise MonoError(rc, "mono_layer_status")
        return rc

    def buffer(self, name: str):
        """(device pointer, bytes) of an intermediate buffer."""
        p, n = C.c_void_p(), C.c_size_t()
        rc = lib().mono_layer_buffer(self._h, BUF[name], C.byref(p), C.byref(n))
        if rc != MONO_OK:
            raise MonoError(rc, "mono_layer_buffer")
        return p.value, n.value

    def read(self, name: str, nbytes: int | None = None):
        """Host copy (numpy uint8) of an intermediate buffer, after the device is idle."""
        import numpy as np
        _, total = self.buffer(name)
        n = total if nbytes is None else nbytes
        out = np.empty(n, np.uint8)
        rc = lib().mono_layer_read_buffer(self._h, BUF[name], out.ctypes.data, n)
        if rc != MONO_OK:
            raise MonoError(rc, "mono_layer_read_buffer")
        return out

    def launches_per_step(self) -> int:
        return lib().mono_layer_launches_per_step(self._h)

    def kernels_last_step(self) -> int:
        """Kernels the last step call on this layer enqueued (empty launch slots excluded)."""
        return lib().mono_layer_kernels_last_step(self._h)

    def launch_names(self) -> list[str]:
        return [lib().mono_layer_launch_name(i).decode() for i in range(self.launches_per_step())]

    def set_profile_events(self, events) -> None:
        """events: list of launches_per_step()+1 torch.cuda.Event (created and recorded once
        so that they exist), or None to stop profiling."""
        if events is None:
            rc = lib().mono_layer_set_profile_events(self._h, None, 0)
        else:
            arr = (C.c_void_p * len(events))(*[e.cuda_event for e in events])
            self._prof = arr
            rc = lib().mono_layer_set_profile_events(self._h, arr, len(events))
        if rc != MONO_OK:
            raise MonoError(rc, "mono_layer_set_profile_events")

    def close(self) -> None:
        if self._h:
            lib().mono_layer_free(self._h)
            self._h = C.c_void_p()

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


__all__ = ["Layer", "MonoError", "lib", "strerror", "make_spec", "Spec", "Weights", "StepArgs",
           "FfnArgs", "BUF", "EXPORTS", "LIB_PATH", "ATTN_WEIGHT_FIELDS"]
