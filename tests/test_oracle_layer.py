"""Pins for the oracle's whole-layer wiring.

The stage functions are pinned in the other oracle tests; here the layer must equal their
composition in launch order, reduce to the residual when the blocks it adds are zeroed,
pass pad rows through, and be sensitive enough that a 3% error in the routed experts fails
the comparison rules.
"""
import copy

import numpy as np
import pytest

import gen
from tests.helpers import bf16_f64, np_inputs
from tests.parity import layer_metrics, layer_ok, near_tie_rows


def _bf16_round(orc, v):
    out = orc.bf16_round_array(v)
    assert np.array_equal(out.ravel()[:50], [orc.bf16_bits(float(x)) for x in np.ravel(v)[:50]])
    return out


@pytest.fixture(scope="module")
def small():
    spec, w, st = gen.make_workload("small_r11")
    wn, sn = np_inputs(w, st)
    return spec, wn, sn


def test_layer_equals_stage_composition(orc, small):
    spec, w, st = small
    tr = orc.layer(spec, w, st)
    assert tr["rc"] == 0
    eps, qr = spec["eps"], spec["q_rank"]
    xn = orc.rmsnorm(st["x"], w["attn_norm"], eps)
    assert np.array_equal(xn, tr["xn"])
    qkv = _bf16_round(orc, orc.gemv_mxfp8(xn, w["wqkv"], w["wqkv_s"]))
    assert np.array_equal(qkv, tr["qkv"])
    qlatn = orc.rmsnorm(qkv[:, :qr], w["q_norm"], eps)
    kvn = orc.rmsnorm(qkv[:, qr:], w["kv_norm"], eps)
    assert np.array_equal(qlatn, tr["q_latn"]) and np.array_equal(kvn, tr["kvn"])
    rc, cache = orc.kv_insert(spec, st, kvn)
    assert rc == 0 and np.array_equal(cache, tr["cache"])
    q = _bf16_round(orc, orc.gemv_mxfp8(qlatn, w["wq_b"], w["wq_b_s"]))
    assert np.array_equal(q, tr["q"])
    rc, o = orc.attention(spec, st, q, cache=cache)
    assert rc == 0 and np.array_equal(o, tr["o"])
    oa = _bf16_round(orc, orc.gemv_mxfp8(o, w["wo_a"], w["wo_a_s"]))
    assert np.array_equal(oa, tr["oa"])
    h = _bf16_round(orc, bf16_f64(st["x"]) + orc.gemv_mxfp8(oa, w["wo_b"], w["wo_b_s"]))
    assert np.array_equal(h, tr["h"])
    u = orc.rmsnorm(h, w["ffn_norm"], eps)
    assert np.array_equal(u, tr["u"])
    rt = orc.router(u, w["router"], spec["topk"], spec["routed_scale"], positions=st["positions"])
    assert np.array_equal(rt["idx"], tr["topk_idx"]) and np.array_equal(rt["w"], tr["topk_w"])
    ts, ys = orc.ffn(u, w["sh_gu"], w["sh_gu_s"], w["sh_d"], w["sh_d_s"], spec["shared_inter"],
                     spec["swiglu_clamp"], fmt4=False)
    assert np.array_equal(ts, tr["t_s"]) and np.array_equal(ys, tr["y_s"])
    yr = np.zeros_like(ys)
    for r in range(u.shape[0]):
        for j, e in enumerate(rt["idx"][r]):
            if e < 0:
                continue
            t1, y1 = orc.ffn(u[r:r + 1], w["ex_gu"][e], w["ex_gu_s"][e], w["ex_d"][e], w["ex_d_s"][e],
                             spec["moe_inter"], spec["swiglu_clamp"], fmt4=True)
            assert np.array_equal(t1[0], tr["t_r"][r, j])
            yr[r] += rt["w"][r, j] * y1[0]
    np.testing.assert_allclose(yr, tr["y_r"], rtol=1e-13, atol=1e-15)
    pad = np.asarray(st["positions"]) < 0
    out = _bf16_round(orc, bf16_f64(h) + ys + tr["y_r"])
    out[pad] = st["x"][pad]
    assert np.array_equal(out, tr["out"])


def test_zero_blocks_reduce_to_residual(orc, small):
    spec, w, st = small
    w0 = dict(w)
    w0["wo_b"] = np.zeros_like(w["wo_b"])          # attention adds nothing: h = x
    w0["sh_gu"] = np.zeros_like(w["sh_gu"])        # shared expert adds nothing
    w0["ex_gu"] = np.zeros_like(w["ex_gu"])        # routed experts add nothing
    tr = orc.layer(spec, w0, st)
    assert np.array_equal(tr["h"], st["x"])
    assert np.array_equal(tr["out"], st["x"])
    assert not tr["y_s"].any() and not tr["y_r"].any()


def test_pad_rows_pass_through(orc, small):
    spec, w, st = small
    tr = orc.layer(spec, w, st)
    pad = np.asarray(st["positions"]) < 0
    assert pad.any()
    assert np.array_equal(tr["out"][pad], st["x"][pad])
    assert (tr["topk_idx"][pad] == -1).all() and not tr["o"][pad].any()


def test_forced_routing(orc, small):
    spec, w, st = small
    tr = orc.layer(spec, w, st)
    same = orc.layer(spec, w, st, force_idx=tr["topk_idx"])
    assert np.array_equal(same["out"], tr["out"])
    other = tr["topk_idx"].copy()
    other[0] = (other[0] + 1) % spec["n_experts"]
    diff = orc.layer(spec, w, st, force_idx=other)
    assert not np.array_equal(diff["out"][0], tr["out"][0])
    assert np.array_equal(diff["out"][1:], tr["out"][1:])


def test_sensitivity_routed_scale_off_by_3_percent_fails(orc, small):
    spec, w, st = small
    valid = np.asarray(st["positions"]) >= 0
    ref = orc.layer(spec, w, st)
    off = orc.layer(dict(spec, routed_scale=1.03), w, st)
    m = layer_metrics(off["out"], ref["out"], off["y_s"], ref["y_s"], off["y_r"], ref["y_r"], valid)
    assert not layer_ok(m), m
    assert m["routed_rel"] > 0.02, m
    m0 = layer_metrics(ref["out"], ref["out"], ref["y_s"], ref["y_s"], ref["y_r"], ref["y_r"], valid)
    assert layer_ok(m0)


def test_noncausal_draft_rows(orc):
    spec, w, st = gen.make_workload("small_r11", causal=0, swa_width=30)
    wn, sn = np_inputs(w, st)
    tr = orc.layer(spec, wn, sn)
    assert tr["rc"] == 0
    # rows of one request attend the same keys -> identical queries would give identical o;
    # here it suffices that every row of a request sees the request's last position
    for r, p in enumerate(sn["positions"]):
        if p < 0:
            continue
        q = sn["row_req"][r]
        e = max(pp for pp, qq in zip(sn["positions"], sn["row_req"]) if qq == q)
        assert orc.key_range(spec, sn, r) == (max(0, e - 29), e)


def test_tiny_layer_runs_and_routes(orc):
    spec, w, st = gen.make_workload("tiny")
    wn, sn = np_inputs(w, st)
    tr = orc.layer(spec, wn, sn)
    assert tr["rc"] == 0
    assert tr["topk_idx"].shape == (1, 2) and len(set(tr["topk_idx"][0])) == 2
    assert np.isclose(tr["topk_w"].sum(), 1.0)
    assert not near_tie_rows(tr["probs"], 2).any()
    assert np.isfinite(bf16_f64(tr["out"])).all()
