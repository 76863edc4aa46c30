"""GPU parity: the CUDA layer (through the C ABI) against the CPU oracle.

For every workload (the tiny oracle case, a ragged mid-size case with a pad row, and the
three full-size shapes: 1 row; 6 non-causal draft rows with top-3; 48 rows with top-6):
  * stage by stage -- each stage's GPU output against the oracle stage evaluated on the
    GPU's own input to that stage (bf16 stages within 1 ulp, KV records bit-exact,
    f32 stages within 1e-4 relative L2, top-k sets equal outside near-ties);
  * end to end -- the GPU layer output against an independent oracle run from the same
    inputs: relative L2 <= 1e-2, cosine >= 0.9997, MoE sum relative L2 <= 1e-2.
"""
import numpy as np
import pytest
import torch

import gen
import oracle
from tests.gpu_harness import check_stages, oracle_threads, routed_sum, run_step, to_device
from tests.helpers import np_inputs
from tests.parity import layer_metrics, layer_ok, near_tie_rows

pytestmark = pytest.mark.gpu

WORKLOADS = ["tiny", "small_r11", "wide_r9", "mid_r13", "skew_r20", "full_r1", "full_r4", "draft_r6",
             "full_r24", "full_r48", "draft_r48"]
_cache = {}


def _need_gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from moe_decode_layer_mxfp8_gb300 import build
    build.build()
    oracle_threads()


def _case(name):
    if name in _cache:
        return _cache[name]
    _need_gpu()
    import moe_decode_layer_mxfp8_gb300 as m
    dev = torch.device("cuda")
    full = gen.WORKLOADS[name]["spec"]["hidden"] >= 4096
    spec, w, st = gen.make_workload(name, weight_device=dev if full else "cpu")
    wd, sd = to_device(w, st, dev)
    wn, sn = np_inputs(w, st)
    layer = m.Layer(spec, wd)
    g = run_step(layer, spec, sd, st["rows"])
    _cache.clear()  # keep at most one full-size case resident
    _cache[name] = (spec, wn, sn, g, layer, wd, sd)
    return _cache[name]


@pytest.mark.parametrize("name", WORKLOADS)
def test_stage_parity(name):
    spec, wn, sn, g, *_ = _case(name)
    assert g["status"] == 0
    res, ties = check_stages(spec, wn, sn, g, sn["x"].shape[0])
    print(name, {k: f"{v:.1e}" for k, v in res.items()}, "near-tie rows:", int(ties.sum()))


@pytest.mark.parametrize("name", WORKLOADS)
def test_layer_matches_oracle(name):
    spec, wn, sn, g, *_ = _case(name)
    valid = np.asarray(sn["positions"]) >= 0
    ref = oracle.layer(spec, wn, sn)
    assert ref["rc"] == 0
    K = spec["topk"]
    ties = near_tie_rows(ref["probs"], K)
    flips = [r for r in np.nonzero(valid)[0]
             if sorted(g["topk_idx"][r]) != sorted(ref["topk_idx"][r])]
    assert all(ties[r] for r in flips), f"routing differs outside near-ties on rows {flips}"
    if flips:  # recompute the MoE with the GPU's choice on the near-tie rows
        forced = ref["topk_idx"].copy()
        forced[flips] = g["topk_idx"][flips]
        ref = oracle.layer(spec, wn, sn, force_idx=forced)
    m = layer_metrics(g["out"], ref["out"], g["y_s"], ref["y_s"], routed_sum(g), ref["y_r"], valid)
    print(name, m, "flipped near-tie rows:", flips)
    assert layer_ok(m), m
    assert np.array_equal(g["cache"], ref["cache"]) or name.startswith("full") or name == "draft_r6" \
        or (g["cache"] != ref["cache"]).sum() <= 8 * spec["kv_dim"]


def test_draft_r48_concentrates_every_row_on_three_experts():
    spec, wn, sn, g, *_ = _case("draft_r48")
    assert (g["topk_idx"] == g["topk_idx"][0]).all()
    assert len(np.unique(g["topk_idx"])) == 3


def test_full_r48_routes_at_least_60_experts():
    spec, wn, sn, g, *_ = _case("full_r48")
    assert len(np.unique(g["topk_idx"])) >= 60


def test_sensitivity_routed_scale_3_percent_fails():
    spec, wn, sn, g, *_ = _case("small_r11")
    valid = np.asarray(sn["positions"]) >= 0
    off = oracle.layer(dict(spec, routed_scale=1.03), wn, sn, force_idx=g["topk_idx"])
    m = layer_metrics(g["out"], off["out"], g["y_s"], off["y_s"], routed_sum(g), off["y_r"], valid)
    assert not layer_ok(m), m
    assert m["routed_rel"] > 0.02, m


def test_replays_are_bit_exact():
    _need_gpu()
    spec, wn, sn, g, layer, wd, sd = _case("small_r11")
    out = torch.empty_like(sd["x"])
    cache = sd["kv_cache"].clone()
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        layer.step(sd["x"], out, sd["positions"], sd["row_req"], sd["block_table"], cache)
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph, stream=s):
            layer.step(sd["x"], out, sd["positions"], sd["row_req"], sd["block_table"], cache)
    torch.cuda.synchronize()
    first = out.clone()
    for _ in range(300):
        graph.replay()
    torch.cuda.synchronize()
    assert torch.equal(out, first)
    assert np.array_equal(first.cpu().view(torch.int16).numpy().view(np.uint16), g["out"])


def test_rows_beyond_max_are_refused():
    _need_gpu()
    import moe_decode_layer_mxfp8_gb300 as m
    spec, wn, sn, g, layer, wd, sd = _case("small_r11")
    x = torch.zeros((layer.max_rows + 1, spec["hidden"]), dtype=torch.bfloat16, device="cuda")
    pos = torch.zeros(layer.max_rows + 1, dtype=torch.int32, device="cuda")
    with pytest.raises(m.MonoError) as e:
        layer.step(x, x, pos, pos, sd["block_table"], sd["kv_cache"])
    assert e.value.code == -3


def test_overlapping_kv_view_is_refused():
    _need_gpu()
    import moe_decode_layer_mxfp8_gb300 as m
    spec, wn, sn, g, layer, wd, sd = _case("small_r11")
    c = sd["kv_cache"]
    bad = c.view(-1)[: c.shape[0] * (c.shape[1] - 1) * c.shape[2]].view(c.shape[0], c.shape[1] - 1, c.shape[2])
    bad = bad.as_strided((c.shape[0], c.shape[1], c.shape[2]), ((c.shape[1] - 1) * c.shape[2], c.shape[2], 1))
    out = torch.empty_like(sd["x"])
    with pytest.raises(m.MonoError) as e:
        layer.step(sd["x"], out, sd["positions"], sd["row_req"], sd["block_table"], bad)
    assert e.value.code == -5


def test_unmapped_page_sets_status_without_fault():
    _need_gpu()
    spec, wn, sn, g, layer, wd, sd = _case("small_r11")
    table = sd["block_table"].clone()
    table[0, :] = 10 ** 6  # outside the cache
    out = torch.empty_like(sd["x"])
    cache = sd["kv_cache"].clone()
    layer.status(clear=True)
    layer.step(sd["x"], out, sd["positions"], sd["row_req"], table, cache)
    torch.cuda.synchronize()
    st = layer.status(clear=True)
    assert st & 1
    assert layer.status() == 0
    # the layer still works afterwards
    layer.step(sd["x"], out, sd["positions"], sd["row_req"], sd["block_table"], cache)
    torch.cuda.synchronize()
    assert layer.status() == 0


def test_handles_with_different_max_rows_coexist():
    """Kernel attributes are process-wide: building a small layer after a large one must not
    break the large one's next step."""
    _need_gpu()
    import moe_decode_layer_mxfp8_gb300 as m
    spec, wn, sn, g, layer, wd, sd = _case("small_r11")
    small = m.Layer(dict(spec, max_rows=1), wd)
    out = torch.empty_like(sd["x"])
    cache = sd["kv_cache"].clone()
    layer.step(sd["x"], out, sd["positions"], sd["row_req"], sd["block_table"], cache)
    torch.cuda.synchronize()
    assert layer.status() == 0
    assert np.array_equal(out.cpu().view(torch.int16).numpy().view(np.uint16), g["out"])
    small.close()


def test_step_in_place_equals_out_of_place():
    """x_out may alias x_in: the layer reads x (norm, residual, pad rows) before the final
    combine overwrites it."""
    _need_gpu()
    spec, wn, sn, g, layer, wd, sd = _case("small_r11")
    x = sd["x"].clone()
    layer.step(x, x, sd["positions"], sd["row_req"], sd["block_table"], sd["kv_cache"].clone())
    torch.cuda.synchronize()
    assert layer.status() == 0
    assert np.array_equal(x.cpu().view(torch.int16).numpy().view(np.uint16), g["out"])


def test_wait_timeout_sets_status_and_leaves_the_context_usable():
    """A bounded pipeline wait that runs out raises the status word's timeout bit and returns;
    the next step runs normally."""
    _need_gpu()
    import moe_decode_layer_mxfp8_gb300 as m
    spec, wn, sn, g, layer, wd, sd = _case("small_r11")
    layer.status(clear=True)
    layer.selftest_wait_timeout(2_000_000)  # 2 ms
    torch.cuda.synchronize()
    assert layer.status(clear=True) & m.STATUS_WAIT_TIMEOUT
    assert layer.status() == 0
    out = torch.empty_like(sd["x"])
    layer.step(sd["x"], out, sd["positions"], sd["row_req"], sd["block_table"], sd["kv_cache"].clone())
    torch.cuda.synchronize()
    assert layer.status() == 0
    assert np.array_equal(out.cpu().view(torch.int16).numpy().view(np.uint16), g["out"])
    with pytest.raises(m.MonoError):
        layer.selftest_wait_timeout(10)  # budget out of range


def test_empty_step_is_refused_and_the_next_step_runs():
    """rows = 0 is outside 1..max_rows: refused before any launch, nothing written."""
    _need_gpu()
    import moe_decode_layer_mxfp8_gb300 as m
    spec, wn, sn, g, layer, wd, sd = _case("small_r11")
    x = torch.zeros((0, spec["hidden"]), dtype=torch.bfloat16, device="cuda")
    pos = torch.zeros(0, dtype=torch.int32, device="cuda")
    cache = sd["kv_cache"].clone()
    with pytest.raises(m.MonoError) as e:
        layer.step(x, x, pos, pos, sd["block_table"], cache)
    assert e.value.code == -1
    torch.cuda.synchronize()
    assert torch.equal(cache, sd["kv_cache"]) and layer.status() == 0
    out = torch.empty_like(sd["x"])
    layer.step(sd["x"], out, sd["positions"], sd["row_req"], sd["block_table"], cache)
    torch.cuda.synchronize()
    assert layer.status() == 0
    assert np.array_equal(out.cpu().view(torch.int16).numpy().view(np.uint16), g["out"])


@pytest.mark.parametrize("name,kernels", [("small_r11", 15), ("full_r48", 14)])
def test_kernels_last_step_counts_the_launched_kernels(name, kernels):
    """Every launch slot runs a kernel at small steps; at large steps the shared expert's
    down GEMM runs inside the routed down launch, so its slot launches nothing."""
    spec, wn, sn, g, layer, wd, sd = _case(name)
    assert layer.launches_per_step() == 15
    run_step(layer, spec, sd, sd["x"].shape[0])
    assert layer.kernels_last_step() == kernels


@pytest.mark.parametrize("name", ["small_r11", "full_r48"])
def test_all_pad_rows_pass_x_through(name):
    """The degenerate step: every row a pad row.  Pad rows leave the layer unchanged
    (out = x, bit for bit), write no KV record and route to no expert (-1, weight 0), so the
    expert GEMMs run with no work item (the clustered small-step and the persistent
    large-step kernels alike)."""
    spec, wn, sn, g, layer, wd, sd = _case(name)
    rows, K = sd["x"].shape[0], spec["topk"]
    pos = torch.full_like(sd["positions"], -1)
    cache = sd["kv_cache"].clone()
    out = torch.empty_like(sd["x"])
    idx = torch.full((rows, K), -7, dtype=torch.int32, device="cuda")
    wts = torch.full((rows, K), 5.0, dtype=torch.float32, device="cuda")
    layer.step(sd["x"], out, pos, sd["row_req"], sd["block_table"], cache,
               topk_idx_out=idx, topk_w_out=wts)
    torch.cuda.synchronize()
    assert layer.status() == 0
    assert torch.equal(out.view(torch.int16), sd["x"].view(torch.int16))
    assert torch.equal(cache, sd["kv_cache"])
    assert (idx == -1).all() and (wts == 0).all()
    # and the handle's next real step is unaffected
    out2 = torch.empty_like(sd["x"])
    layer.step(sd["x"], out2, sd["positions"], sd["row_req"], sd["block_table"], cache)
    torch.cuda.synchronize()
    assert layer.status() == 0
    assert np.array_equal(out2.cpu().view(torch.int16).numpy().view(np.uint16), g["out"])


def test_f16_operand_overflow_saturates_and_raises_status():
    """wo_a's E8M0 block scales raised by 2^20: its output oa (copied to f16 as wo_b's
    tensor-core operand) then lies far beyond f16's range.  The copies saturate at +-65504
    and raise MONO_STATUS_F16_RANGE instead of becoming infinities; the step's output stays
    finite and the next normal step is unaffected."""
    _need_gpu()
    import moe_decode_layer_mxfp8_gb300 as m
    spec, wn, sn, g, layer, wd, sd = _case("small_r11")
    big = dict(wd)
    big["wo_a_s"] = (wd["wo_a_s"].to(torch.int32) + 20).clamp(max=254).to(torch.uint8)
    loud = m.Layer(spec, big)
    out = torch.empty_like(sd["x"])
    loud.step(sd["x"], out, sd["positions"], sd["row_req"], sd["block_table"], sd["kv_cache"].clone())
    torch.cuda.synchronize()
    st = loud.status(clear=True)
    assert st & m.STATUS_F16_RANGE, st
    rows, o_rank = sn["x"].shape[0], spec["o_rank"]
    oa = loud.read("oa", rows * o_rank * 2).view(np.float16).reshape(rows, o_rank).astype(np.float32)
    live = np.asarray(sn["positions"]) >= 0
    assert np.isfinite(oa).all()
    assert np.abs(oa[live]).max() == 65504.0
    assert torch.isfinite(out.float()).all()
    loud.close()
    # the ordinary layer: no flag
    out2 = torch.empty_like(sd["x"])
    layer.status(clear=True)
    layer.step(sd["x"], out2, sd["positions"], sd["row_req"], sd["block_table"], sd["kv_cache"].clone())
    torch.cuda.synchronize()
    assert layer.status() == 0
