"""GPU-test plumbing: run one layer step through the C ABI and collect every stage's output,
then compare each stage with the oracle evaluated on the GPU's own input to that stage."""
from __future__ import annotations

import os

import numpy as np
import torch

import oracle
from tests.helpers import bf16_f64, np_inputs, rel_l2


def f16_to_bf16_bits(a: np.ndarray) -> np.ndarray:
    """f16 copies of bf16 values back to bf16 bit patterns (exact for in-range values)."""
    return torch.from_numpy(np.ascontiguousarray(a).astype(np.float32)).to(torch.bfloat16).view(
        torch.int16).numpy().view(np.uint16)


def to_device(w: dict, st: dict, dev):
    wd = {k: v.to(dev) for k, v in w.items()}
    sd = {k: (v.to(dev) if isinstance(v, torch.Tensor) else v) for k, v in st.items()}
    return wd, sd


def run_step(layer, spec, sd, rows, x_out=None):
    """One step on a private copy of the cache; returns host copies of everything."""
    import moe_decode_layer_mxfp8_gb300 as m  # noqa: F401  (the layer object carries the lib)
    dev = sd["x"].device
    cache = sd["kv_cache"].clone()
    out = torch.empty_like(sd["x"]) if x_out is None else x_out
    K = spec["topk"]
    idx = torch.full((rows, K), -7, dtype=torch.int32, device=dev)
    wts = torch.zeros((rows, K), dtype=torch.float32, device=dev)
    layer.step(sd["x"], out, sd["positions"], sd["row_req"], sd["block_table"], cache,
               topk_idx_out=idx, topk_w_out=wts)
    torch.cuda.synchronize()
    H, E, I, Is = spec["hidden"], spec["n_experts"], spec["moe_inter"], spec["shared_inter"]
    QW, A = spec["n_q_heads"] * spec["head_dim"], spec["q_rank"] + spec["kv_dim"]

    def rd(name, dtype, shape):
        n = int(np.prod(shape)) * np.dtype(dtype).itemsize
        return layer.read(name, n).view(dtype).reshape(shape)

    g = dict(
        status=layer.status(),
        out=out.cpu().view(torch.int16).numpy().view(np.uint16),
        cache=cache.cpu().numpy(),
        user_idx=idx.cpu().numpy(), user_w=wts.cpu().numpy(),
        xn=f16_to_bf16_bits(rd("xn", np.float16, (rows, H))),
        qkv=rd("qkv", np.uint16, (rows, A)),
        q_latn=f16_to_bf16_bits(rd("qlatn", np.float16, (rows, spec["q_rank"]))),
        kvn=rd("kvn", np.uint16, (rows, spec["kv_dim"])),
        q=rd("q", np.uint16, (rows, QW)),
        o=f16_to_bf16_bits(rd("o", np.float16, (rows, QW))),
        oa=f16_to_bf16_bits(rd("oa", np.float16, (rows, spec["o_rank"]))),
        h=rd("h", np.uint16, (rows, H)),
        u=f16_to_bf16_bits(rd("u", np.float16, (rows, H))),
        logits=rd("logits", np.float32, (rows, E)),
        topk_idx=rd("topk_idx", np.int32, (rows, K)),
        topk_w=rd("topk_w", np.float32, (rows, K)),
        slot_pos=rd("slot_pos", np.int32, (rows, K)),
        t_s=f16_to_bf16_bits(rd("ts", np.float16, (rows, Is))),
        y_s=rd("ys", np.float32, (rows, H)),
        t_r=f16_to_bf16_bits(rd("tr", np.float16, (rows * K, I))),
        y_r=rd("yr", np.float32, (rows * K, H)),
    )
    return g


def run_ffn_step(layer, spec, x, attn, positions, x_out=None):
    """One FFN launch; returns host copies of its output and of the MoE-half buffers."""
    dev = x.device
    rows = x.shape[0]
    out = torch.empty_like(x) if x_out is None else x_out
    K = spec["topk"]
    idx = torch.full((rows, K), -7, dtype=torch.int32, device=dev)
    wts = torch.zeros((rows, K), dtype=torch.float32, device=dev)
    layer.ffn_step(x, attn, out, positions, topk_idx_out=idx, topk_w_out=wts)
    torch.cuda.synchronize()
    H, E, I, Is = spec["hidden"], spec["n_experts"], spec["moe_inter"], spec["shared_inter"]

    def rd(name, dtype, shape):
        n = int(np.prod(shape)) * np.dtype(dtype).itemsize
        return layer.read(name, n).view(dtype).reshape(shape)

    return dict(
        status=layer.status(),
        out=out.cpu().view(torch.int16).numpy().view(np.uint16),
        user_idx=idx.cpu().numpy(), user_w=wts.cpu().numpy(),
        h=rd("h", np.uint16, (rows, H)),
        u=f16_to_bf16_bits(rd("u", np.float16, (rows, H))),
        logits=rd("logits", np.float32, (rows, E)),
        topk_idx=rd("topk_idx", np.int32, (rows, K)),
        topk_w=rd("topk_w", np.float32, (rows, K)),
        slot_pos=rd("slot_pos", np.int32, (rows, K)),
        t_s=f16_to_bf16_bits(rd("ts", np.float16, (rows, Is))),
        y_s=rd("ys", np.float32, (rows, H)),
        t_r=f16_to_bf16_bits(rd("tr", np.float16, (rows * K, I))),
        y_r=rd("yr", np.float32, (rows * K, H)),
    )


def routed_sum(g):
    """sum_j w_j y_j per row from the GPU's buffers."""
    out = np.zeros(g["y_s"].shape, np.float64)
    for r in range(out.shape[0]):
        for j, pos in enumerate(g["slot_pos"][r]):
            if pos >= 0:
                out[r] += float(g["topk_w"][r, j]) * g["y_r"][pos].astype(np.float64)
    return out


def moe_sum(g):
    """y_shared + sum_j w_j y_j from the GPU's buffers."""
    return g["y_s"].astype(np.float64) + routed_sum(g)


# ---------------------------------------------------------------------------- comparisons
def bf16_ulp_check(got_bits, want_bits, name, ulps=1, rel_floor=2e-3):
    """Elementwise: |got - want| <= ulps * ulp(max(|got|, |want|)) + rel_floor * rms(want)."""
    g, w = bf16_f64(got_bits), bf16_f64(want_bits)
    mag = np.maximum(np.abs(g), np.abs(w))
    e = np.floor(np.log2(np.where(mag > 0, mag, 1.0)))
    ulp = np.exp2(e - 7)
    rms = float(np.sqrt(np.mean(w ** 2))) if w.size else 0.0
    bad = np.abs(g - w) > ulps * ulp + rel_floor * rms
    assert not bad.any(), (f"{name}: {int(bad.sum())}/{bad.size} elements off by more than "
                           f"{ulps} ulp; worst {np.abs(g - w).max():.3e}; rel_l2 {rel_l2(g, w):.2e}")
    return rel_l2(g, w)


def f32_check(got, want, name, rel=1e-4, abs_frac=2e-3):
    got, want = np.asarray(got, np.float64), np.asarray(want, np.float64)
    r = rel_l2(got, want)
    rms = float(np.sqrt(np.mean(want ** 2))) if want.size else 0.0
    worst = float(np.abs(got - want).max()) if want.size else 0.0
    assert r <= rel and worst <= abs_frac * rms + 1e-30, f"{name}: rel_l2 {r:.2e}, worst {worst:.2e}, rms {rms:.2e}"
    return r


def _round(v):
    return oracle.bf16_round_array(v)


def check_stages(spec, wn, sn, g, rows):
    """Every stage of the GPU step against the oracle stage on the GPU's own stage input."""
    valid = np.asarray(sn["positions"]) >= 0
    eps, qr, K = spec["eps"], spec["q_rank"], spec["topk"]
    res = {}
    res["xn"] = bf16_ulp_check(g["xn"], oracle.rmsnorm(sn["x"], wn["attn_norm"], eps), "xn")
    res["qkv"] = bf16_ulp_check(g["qkv"], _round(oracle.gemv_mxfp8(g["xn"], wn["wqkv"], wn["wqkv_s"])), "qkv")
    res["q_latn"] = bf16_ulp_check(g["q_latn"], oracle.rmsnorm(g["qkv"][:, :qr], wn["q_norm"], eps), "q_latn")
    res["kvn"] = bf16_ulp_check(g["kvn"], oracle.rmsnorm(g["qkv"][:, qr:], wn["kv_norm"], eps), "kvn")
    rc, cache_want = oracle.kv_insert(spec, sn, g["kvn"])
    assert rc == 0
    diff = np.nonzero(g["cache"] != cache_want)
    assert diff[0].size == 0, f"KV cache differs at {diff[0].size} bytes, first at {tuple(d[0] for d in diff)}"
    res["q"] = bf16_ulp_check(g["q"], _round(oracle.gemv_mxfp8(g["q_latn"], wn["wq_b"], wn["wq_b_s"])), "q")
    rc, o_want = oracle.attention(spec, sn, g["q"], cache=g["cache"])
    assert rc == 0
    res["o"] = bf16_ulp_check(g["o"], o_want, "o")
    res["oa"] = bf16_ulp_check(g["oa"], _round(oracle.gemv_mxfp8(g["o"], wn["wo_a"], wn["wo_a_s"])), "oa")
    h_want = _round(bf16_f64(sn["x"]) + oracle.gemv_mxfp8(g["oa"], wn["wo_b"], wn["wo_b_s"]))
    res["h"] = bf16_ulp_check(g["h"], h_want, "h")
    ties = check_moe(spec, wn, sn["x"], sn["positions"], g, res)
    return res, ties


def check_moe(spec, wn, x, positions, g, res):
    """The FFN seam and MoE stages (u .. out) against the oracle stages on the GPU's own
    inputs; returns the near-tie rows of the routing."""
    valid = np.asarray(positions) >= 0
    eps, K = spec["eps"], spec["topk"]
    res["u"] = bf16_ulp_check(g["u"], oracle.rmsnorm(g["h"], wn["ffn_norm"], eps), "u")
    rt = oracle.router(g["u"], wn["router"], K, spec["routed_scale"], positions=positions)
    res["logits"] = f32_check(g["logits"][valid], rt["logits"][valid], "logits", rel=1e-5)
    from tests.parity import topk_agree
    ok, ties = topk_agree(g["topk_idx"], rt["idx"], rt["probs"], K, valid)
    assert ok, "top-k sets differ on rows without a near-tie"
    assert np.array_equal(g["user_idx"], g["topk_idx"]) and np.array_equal(g["user_w"], g["topk_w"])
    assert (g["topk_idx"][~valid] == -1).all()
    # weights: for the GPU's own indices, the renormalised probabilities of the GPU logits
    for r in np.nonzero(valid)[0]:
        z = g["logits"][r].astype(np.float64)[g["topk_idx"][r]]
        p = np.exp(z - z.max())
        np.testing.assert_allclose(g["topk_w"][r], p / p.sum() * spec["routed_scale"], rtol=2e-6, atol=1e-7)
    # grouping: slot_pos is a bijection onto the sorted positions, grouped by expert
    pos = g["slot_pos"][valid].ravel()
    assert sorted(pos.tolist()) == list(range(pos.size))
    ex_sorted = np.empty(pos.size, np.int64)
    ex_sorted[pos] = g["topk_idx"][valid].ravel()
    assert (np.diff(ex_sorted) >= 0).all()
    # shared expert
    t_s, _ = oracle.ffn(g["u"], wn["sh_gu"], wn["sh_gu_s"], wn["sh_d"], wn["sh_d_s"],
                        spec["shared_inter"], spec["swiglu_clamp"], fmt4=False)
    res["t_s"] = bf16_ulp_check(g["t_s"], t_s, "t_s")
    ys_want = oracle.gemv_mxfp8(g["t_s"], wn["sh_d"], wn["sh_d_s"])
    res["y_s"] = f32_check(g["y_s"], ys_want, "y_s")
    # routed experts, one expert at a time on the rows the GPU routed to it
    I = spec["moe_inter"]
    tr_g, yr_g, tr_w, yr_w = [], [], [], []
    for e in np.unique(g["topk_idx"][valid]):
        sel = [(r, j) for r in np.nonzero(valid)[0] for j in range(K) if g["topk_idx"][r, j] == e]
        ps = [g["slot_pos"][r, j] for r, j in sel]
        u_rows = np.stack([g["u"][r] for r, _ in sel])
        t_e, _ = oracle.ffn(u_rows, wn["ex_gu"][e], wn["ex_gu_s"][e], wn["ex_d"][e], wn["ex_d_s"][e],
                            I, spec["swiglu_clamp"], fmt4=True)
        y_e = oracle.gemv_mxfp4(g["t_r"][ps], wn["ex_d"][e], wn["ex_d_s"][e])
        tr_g.append(g["t_r"][ps]), tr_w.append(t_e), yr_g.append(g["y_r"][ps]), yr_w.append(y_e)
    res["t_r"] = bf16_ulp_check(np.concatenate(tr_g), np.concatenate(tr_w), "t_r")
    res["y_r"] = f32_check(np.concatenate(yr_g), np.concatenate(yr_w), "y_r")
    # final combine
    out_want = _round(bf16_f64(g["h"]) + moe_sum(g))
    out_want[~valid] = x[~valid]
    res["out"] = bf16_ulp_check(g["out"], out_want, "out")
    assert np.array_equal(g["out"][~valid], x[~valid])
    return ties


def oracle_threads():
    oracle.set_threads(max(1, os.cpu_count() or 1))
