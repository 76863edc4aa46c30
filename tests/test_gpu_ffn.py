"""GPU parity of the FFN launch (the residual from an attention output, then the FFN seam and
the MoE) through the C ABI, against the CPU oracle.

For each workload the step's rows get an attention output drawn by ``gen.make_attn_out``:
  * the residual h = bf16(x + a) bit-exact, then every MoE stage against the oracle stage on
    the GPU's own input to it (the same bars as the whole-layer stage checks);
  * end to end against the oracle's FFN launch from the same inputs: relative L2 <= 1e-2,
    cosine >= 0.9997, MoE sum relative L2 <= 1e-2, routing equal outside near-ties;
  * an FFN-only handle (built without attention weights) gives the same bits as a full one,
    and refuses the whole-layer step;
  * the FFN launch fed the whole layer's residual with a -0 attention output reproduces the
    layer's output bit for bit (the two share their kernels);
  * the whole layer and the FFN launch captured in one CUDA graph, 48-row and 6-row steps
    alternating, replay bit-exactly 1,000 times.
"""
import numpy as np
import pytest
import torch

import gen
import oracle
from tests.gpu_harness import (check_moe, oracle_threads, routed_sum, run_ffn_step, run_step,
                               to_device)
from tests.helpers import bf16_f64, np_inputs
from tests.parity import layer_metrics, layer_ok, near_tie_rows

pytestmark = pytest.mark.gpu

WORKLOADS = ["tiny", "small_r11", "wide_r9", "mid_r13", "skew_r20", "full_r1", "full_r24",
             "full_r48"]
_cache = {}


def _need_gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from moe_decode_layer_mxfp8_gb300 import build
    build.build()
    oracle_threads()


def _bits(t):
    return t.cpu().view(torch.int16).numpy().view(np.uint16)


def _case(name):
    if name in _cache:
        return _cache[name]
    _need_gpu()
    import moe_decode_layer_mxfp8_gb300 as m
    dev = torch.device("cuda")
    full = gen.WORKLOADS[name]["spec"]["hidden"] >= 4096
    spec, w, st = gen.make_workload(name, weight_device=dev if full else "cpu")
    a = gen.make_attn_out(spec, st, seed=gen.WORKLOADS[name]["seed"])
    wd, sd = to_device(w, st, dev)
    wn, sn = np_inputs(w, st)
    an = _bits(a)
    ad = a.to(dev)
    ffn_w = {k: v for k, v in wd.items() if k not in m.ATTN_WEIGHT_FIELDS}
    layer = m.Layer(spec, ffn_w)
    g = run_ffn_step(layer, spec, sd["x"], ad, sd["positions"])
    _cache.clear()  # keep at most one full-size case resident
    _cache[name] = (spec, wn, sn, an, g, layer, wd, sd, ad)
    return _cache[name]


@pytest.mark.parametrize("name", WORKLOADS)
def test_ffn_stage_parity(name):
    spec, wn, sn, an, g, *_ = _case(name)
    assert g["status"] == 0
    h_want = oracle.bf16_round_array(bf16_f64(sn["x"]) + bf16_f64(an))
    assert np.array_equal(g["h"], h_want)
    res = {}
    ties = check_moe(spec, wn, sn["x"], sn["positions"], g, res)
    assert np.array_equal(g["user_idx"], g["topk_idx"]) and np.array_equal(g["user_w"], g["topk_w"])
    print(name, {k: f"{v:.1e}" for k, v in res.items()}, "near-tie rows:", int(ties.sum()))


@pytest.mark.parametrize("name", WORKLOADS)
def test_ffn_matches_oracle(name):
    spec, wn, sn, an, g, *_ = _case(name)
    valid = np.asarray(sn["positions"]) >= 0
    ref = oracle.ffn_layer(spec, wn, sn["x"], an, sn["positions"])
    ties = near_tie_rows(ref["probs"], spec["topk"])
    flips = [r for r in np.nonzero(valid)[0] if sorted(g["topk_idx"][r]) != sorted(ref["topk_idx"][r])]
    assert all(ties[r] for r in flips), f"routing differs outside near-ties on rows {flips}"
    if flips:
        forced = ref["topk_idx"].copy()
        forced[flips] = g["topk_idx"][flips]
        ref = oracle.ffn_layer(spec, wn, sn["x"], an, sn["positions"], force_idx=forced)
    m = layer_metrics(g["out"], ref["out"], g["y_s"], ref["y_s"], routed_sum(g), ref["y_r"], valid)
    print(name, m, "flipped near-tie rows:", flips)
    assert layer_ok(m), m
    assert np.array_equal(g["out"][~valid], sn["x"][~valid])


def test_ffn_only_handle_equals_full_handle():
    _need_gpu()
    import moe_decode_layer_mxfp8_gb300 as m
    spec, wn, sn, an, g, ffn_layer, wd, sd, ad = _case("small_r11")
    full = m.Layer(spec, wd)
    g2 = run_ffn_step(full, spec, sd["x"], ad, sd["positions"])
    for k in ("out", "h", "u", "topk_idx", "topk_w", "y_s", "y_r"):
        assert np.array_equal(g2[k], g[k]), k
    full.close()
    out = torch.empty_like(sd["x"])
    with pytest.raises(m.MonoError) as e:
        ffn_layer.step(sd["x"], out, sd["positions"], sd["row_req"], sd["block_table"], sd["kv_cache"])
    assert e.value.code == -1


@pytest.mark.parametrize("name", ["small_r11", "full_r48"])
def test_ffn_launch_reproduces_layer_moe_half(name):
    _need_gpu()
    import moe_decode_layer_mxfp8_gb300 as m
    spec, wn, sn, an, g, ffn_layer, wd, sd, ad = _case(name)
    full = m.Layer(spec, wd)
    lay = run_step(full, spec, sd, sn["x"].shape[0])
    h = torch.from_numpy(lay["h"].view(np.int16)).view(torch.bfloat16).cuda()
    minus_zero = torch.full_like(h, -0.0)  # x + (-0) = x for every x, signed zeros included
    got = run_ffn_step(full, spec, h, minus_zero, sd["positions"])
    valid = np.asarray(sn["positions"]) >= 0
    assert np.array_equal(got["h"], lay["h"])
    for k in ("u", "logits", "topk_idx", "topk_w", "y_s"):
        assert np.array_equal(got[k], lay[k]), k
    assert np.array_equal(got["out"][valid], lay["out"][valid])
    full.close()


def test_layer_and_ffn_launch_in_one_graph_replay_bit_exactly():
    """48-row and 6-row steps alternating, whole layers and FFN launches in one graph; every
    output of 1,000 replays equals the first run's bit for bit."""
    _need_gpu()
    import moe_decode_layer_mxfp8_gb300 as m
    dev = torch.device("cuda")
    spec, w, st = gen.make_workload("full_r48", weight_device=dev)
    wd, sd = to_device(w, st, dev)
    a = gen.make_attn_out(spec, st, seed=3).to(dev)
    lay = m.Layer(spec, wd)
    ffn = m.Layer(spec, {k: v for k, v in wd.items() if k not in m.ATTN_WEIGHT_FIELDS})
    cache = sd["kv_cache"].clone()
    rows6 = slice(0, 6)
    bufs = [torch.empty_like(sd["x"]) for _ in range(4)]
    small = [torch.empty_like(sd["x"][rows6]) for _ in range(2)]

    def step():
        lay.step(sd["x"], bufs[0], sd["positions"], sd["row_req"], sd["block_table"], cache)
        ffn.ffn_step(bufs[0], a, bufs[1], sd["positions"])
        lay.step(sd["x"][rows6], small[0], sd["positions"][rows6], sd["row_req"][rows6],
                 sd["block_table"], cache)
        ffn.ffn_step(small[0], a[rows6], small[1], sd["positions"][rows6])
        lay.step(bufs[1], bufs[2], sd["positions"], sd["row_req"], sd["block_table"], cache)
        ffn.ffn_step(bufs[2], a, bufs[3], sd["positions"])

    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        step()
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph, stream=s):
            step()
    torch.cuda.synchronize()
    first = [b.clone() for b in bufs + small]
    for _ in range(10):  # checked every 100 replays
        for _ in range(100):
            graph.replay()
        torch.cuda.synchronize()
        for b, f in zip(bufs + small, first):
            assert torch.equal(b, f)
    assert lay.status() == 0 and ffn.status() == 0
    assert torch.isfinite(bufs[3].float()).all()
    lay.close(), ffn.close()


@pytest.mark.parametrize("alias", ["x_in", "attn_in"])
def test_ffn_output_may_alias_an_input(alias):
    _need_gpu()
    spec, wn, sn, an, g, layer, wd, sd, ad = _case("small_r11")
    x, a = sd["x"].clone(), ad.clone()
    out = x if alias == "x_in" else a
    layer.ffn_step(x, a, out, sd["positions"])
    torch.cuda.synchronize()
    assert layer.status() == 0
    assert np.array_equal(_bits(out), g["out"])


def test_empty_ffn_launch_is_refused():
    _need_gpu()
    import moe_decode_layer_mxfp8_gb300 as m
    spec, wn, sn, an, g, layer, wd, sd, ad = _case("small_r11")
    x = torch.zeros((0, spec["hidden"]), dtype=torch.bfloat16, device="cuda")
    pos = torch.zeros(0, dtype=torch.int32, device="cuda")
    with pytest.raises(m.MonoError) as e:
        layer.ffn_step(x, x, x, pos)
    assert e.value.code == -1
    assert layer.status() == 0


@pytest.mark.parametrize("name", ["small_r11", "full_r48"])
def test_all_pad_ffn_launch_passes_x_through(name):
    """Every row a pad row: the FFN launch returns x_in unchanged (the attention output is
    not added on pad rows), routes to no expert and leaves the handle usable."""
    spec, wn, sn, an, g, layer, wd, sd, ad = _case(name)
    rows, K = sd["x"].shape[0], spec["topk"]
    pos = torch.full_like(sd["positions"], -1)
    out = torch.empty_like(sd["x"])
    idx = torch.full((rows, K), -7, dtype=torch.int32, device="cuda")
    wts = torch.full((rows, K), 5.0, dtype=torch.float32, device="cuda")
    layer.ffn_step(sd["x"], ad, out, pos, topk_idx_out=idx, topk_w_out=wts)
    torch.cuda.synchronize()
    assert layer.status() == 0
    assert torch.equal(out.view(torch.int16), sd["x"].view(torch.int16))
    assert (idx == -1).all() and (wts == 0).all()
    layer.ffn_step(sd["x"], ad, out, sd["positions"])
    torch.cuda.synchronize()
    assert layer.status() == 0
    assert np.array_equal(_bits(out), g["out"])
