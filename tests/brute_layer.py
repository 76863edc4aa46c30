"""Independent f64 brute force of one decode-layer step, in NumPy -- TEST INFRASTRUCTURE.

A second, separately written restatement of what the layer computes, used to pin the C
oracle (``oracle/oracle.c``).  It shares no code with the oracle (nor with the CUDA path):
its own MX decode (the OCP e2m1 magnitude table, torch's float8_e4m3fn decode for e4m3,
2^(e-127) for E8M0), its own bf16 rounding (round-to-nearest-even by masking the low bits of
the f64 representation), and a different evaluation structure (dense dequantised matrices
and per-row, per-slot loops where the oracle groups rows by expert).

The layer ("Mono decode layer for DeepSeek-V4.1-Flash on MI355X", section Purpose, launch
table rows K1 and K2; draft layers in "Mono decode for the DSpark draft layers", section
Details), with the readings the pages leave open:
  A1 xn = RMSNorm(x) * attn_norm                         rounded to bf16
  A2 qkv = xn . Wqkv^T                                   rounded to bf16
  A3 q_latn = RMSNorm(q latent) * q_norm, kvn = RMSNorm(kv) * kv_norm      bf16
  A4 record of kvn at the row's position: s = amax / 448 (1 if amax = 0) in f32,
     codes = e4m3(kvn / s) in f32, nearest even, saturating; pad rows write nothing
  A5 q = q_latn . Wq_b^T                                 bf16
  B1-B2 per head h: keys/values = the cached latent's slice h / (n_q / slices) over the
     row's window, o_h = softmax(q_h . k_t / sqrt(head_dim)) . v_t   bf16; pad rows 0
  B3 oa = o . Wo_a^T                                     bf16
  B4 h = x + oa . Wo_b^T                                 bf16
  B5 u = RMSNorm(h) * ffn_norm                           bf16
  B6 z = u . Wr^T rounded to f32, p = softmax(z); top-k by z, ties to the lower expert;
     w_j = p_j / sum of the chosen p, times routed_scale; pad rows route nowhere
  B8 shared: t = silu(clamp(g)) * clamp(up) in bf16 (gate rows first), y_s = t . Wd^T
  B9 routed: per (row, slot): the same expert MLP with MXFP4 weights, y_r = sum_j w_j y_j
  B10 out = h + y_s + y_r                                bf16; pad rows out = x
Rounding happens only at the points marked bf16 (and the f32 logits / KV scale).
"""
from __future__ import annotations

import math

import numpy as np
import torch

# OCP Microscaling v1.0, e2m1: magnitudes of the 3-bit code, bit 3 is the sign
E2M1_MAGNITUDE = np.array([0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0])


# ---------------------------------------------------------------------------- formats
def bf16_value(bits) -> np.ndarray:
    b = np.asarray(bits, np.uint16).astype(np.uint32) << 16
    return b.view(np.float32).astype(np.float64)


def bf16_rne(v) -> np.ndarray:
    """f64 values -> bf16 bit patterns, round to nearest even, by masking the f64 bits:
    bf16 keeps 7 of the 52 explicit mantissa bits.  Normal range only (the layer's values
    are far from bf16's subnormals and overflow)."""
    v = np.asarray(v, np.float64)
    u = v.view(np.uint64)
    drop = np.uint64(45)
    half = np.uint64(1) << np.uint64(44)
    lsb = (u >> drop) & np.uint64(1)
    r = (u + (half - np.uint64(1)) + lsb) & ~((np.uint64(1) << drop) - np.uint64(1))
    r = np.where(v == 0.0, u, r)  # keep signed zeros
    f32 = r.view(np.float64).astype(np.float32)  # exact: 8 significant bits
    return (f32.view(np.uint32) >> np.uint32(16)).astype(np.uint16)


def e4m3_value(codes) -> np.ndarray:
    t = torch.from_numpy(np.ascontiguousarray(np.asarray(codes, np.uint8)))
    return t.view(torch.float8_e4m3fn).to(torch.float64).numpy()


def e4m3_encode_f32(v32: np.ndarray) -> np.ndarray:
    """f32 values -> e4m3 codes, nearest even, saturating at +-448 (torch's cast after a clamp)."""
    t = torch.from_numpy(np.clip(np.asarray(v32, np.float32), -448.0, 448.0))
    return t.to(torch.float8_e4m3fn).view(torch.uint8).numpy()


def e8m0_value(codes) -> np.ndarray:
    return np.ldexp(1.0, np.asarray(codes, np.int64) - 127)


def dequant_mxfp8(codes, scales) -> np.ndarray:
    """[N, K] e4m3 with one E8M0 scale per 32x32 block -> f64 [N, K]."""
    w = e4m3_value(codes)
    s = e8m0_value(scales)
    return w * np.repeat(np.repeat(s, 32, axis=0), 32, axis=1)


def dequant_mxfp4(packed, scales) -> np.ndarray:
    """[N, K/2] packed e2m1 (element 2i in the low nibble) with one scale per row and 32
    elements -> f64 [N, K]."""
    p = np.asarray(packed, np.uint8)
    nib = np.empty(p.shape[:-1] + (2 * p.shape[-1],), np.uint8)
    nib[..., 0::2] = p & 0xF
    nib[..., 1::2] = p >> 4
    mag = E2M1_MAGNITUDE[nib & 7]
    val = np.where(nib & 8, -mag, mag)
    return val * np.repeat(e8m0_value(scales), 32, axis=-1)


# ----------------------------------------------------------------------------- stages
def rmsnorm_bits(x_bits, gamma_bits, eps) -> np.ndarray:
    x = bf16_value(x_bits)
    ms = np.mean(x * x, axis=-1, keepdims=True)
    return bf16_rne(x / np.sqrt(ms + float(np.float32(eps))) * bf16_value(gamma_bits))


def swiglu_clamped(g, u, c):
    g = np.clip(g, -c, c)
    u = np.clip(u, -c, c)
    return g / (1.0 + np.exp(-g)) * u


def key_window(spec, positions, row_req, r):
    """(lo, hi) inclusive positions row r attends, or None for a pad row."""
    p = int(positions[r])
    if p < 0:
        return None
    if spec["causal"]:
        hi, width = p, spec["window"]
    else:
        hi = max(int(q) for q, rq in zip(positions, row_req) if rq == row_req[r])
        width = spec["swa_width"]
    return max(0, hi - width + 1), hi


def record(cache, block_table, block_size, req, t):
    return cache[block_table[req, t // block_size], t % block_size]


def attention_row(spec, q_row_f64, cache, block_table, req, lo, hi) -> np.ndarray:
    """o (f64, unrounded) of one row: per head softmax(q.k / sqrt(head_dim)) . v."""
    nq, dh, kvd, bs = spec["n_q_heads"], spec["head_dim"], spec["kv_dim"], spec["block_size"]
    groups = kvd // dh
    lat = []
    for t in range(lo, hi + 1):
        rec = record(cache, block_table, bs, req, t)
        scale = float(np.frombuffer(rec[kvd:kvd + 4].tobytes(), np.float32)[0])
        lat.append(e4m3_value(rec[:kvd]) * scale)
    lat = np.stack(lat)                                  # [T, kv_dim]: key = value
    out = np.zeros(nq * dh)
    for h in range(nq):
        g = h // (nq // groups)
        kv = lat[:, g * dh:(g + 1) * dh]
        s = kv @ q_row_f64[h * dh:(h + 1) * dh] / math.sqrt(dh)
        e = np.exp(s - s.max())
        out[h * dh:(h + 1) * dh] = (e / e.sum()) @ kv
    return out


def topk_route(z32_row, k, routed_scale):
    z = z32_row.astype(np.float64)
    p = np.exp(z - z.max())
    p /= p.sum()
    order = np.argsort(-z32_row, kind="stable")[:k]      # ties keep the lower expert
    w = p[order] / p[order].sum() * routed_scale
    return order.astype(np.int32), w, p


# ------------------------------------------------------------------------------ layer
def layer(spec: dict, w: dict, st: dict) -> dict:
    """One step on numpy inputs (bf16 as uint16 bits, as gen.make_workload / np_inputs give
    them).  Returns every stage (bf16 bits, or f64 / f32 / int where the layer keeps those)
    and the cache after the insert."""
    H, nq, dh = spec["hidden"], spec["n_q_heads"], spec["head_dim"]
    qr, kvd, E, K = spec["q_rank"], spec["kv_dim"], spec["n_experts"], spec["topk"]
    I, eps, clamp = spec["moe_inter"], spec["eps"], float(spec["swiglu_clamp"])
    bs = spec["block_size"]
    x = np.asarray(st["x"], np.uint16)
    pos = np.asarray(st["positions"]).astype(np.int64)
    req = np.asarray(st["row_req"]).astype(np.int64)
    table = np.asarray(st["block_table"]).astype(np.int64)
    R = x.shape[0]
    cache = np.array(st["kv_cache"], np.uint8, copy=True)

    xn = rmsnorm_bits(x, w["attn_norm"], eps)                                         # A1
    qkv = bf16_rne(bf16_value(xn) @ dequant_mxfp8(w["wqkv"], w["wqkv_s"]).T)          # A2
    q_latn = rmsnorm_bits(qkv[:, :qr], w["q_norm"], eps)                              # A3
    kvn = rmsnorm_bits(qkv[:, qr:], w["kv_norm"], eps)
    for r in range(R):                                                                # A4
        if pos[r] < 0:
            continue
        v32 = bf16_value(kvn[r]).astype(np.float32)
        amax = np.float32(np.max(np.abs(v32)))
        s = np.float32(amax / np.float32(448.0)) if amax > 0 else np.float32(1.0)
        rec = record(cache, table, bs, req[r], pos[r])
        rec[:kvd] = e4m3_encode_f32(v32 / s)
        rec[kvd:kvd + 4] = np.frombuffer(np.float32(s).tobytes(), np.uint8)
    q = bf16_rne(bf16_value(q_latn) @ dequant_mxfp8(w["wq_b"], w["wq_b_s"]).T)        # A5
    o_f = np.zeros((R, nq * dh))                                                      # B1-B2
    for r in range(R):
        win = key_window(spec, pos, req, r)
        if win is not None:
            o_f[r] = attention_row(spec, bf16_value(q[r]), cache, table, req[r], *win)
    o = bf16_rne(o_f)
    oa = bf16_rne(bf16_value(o) @ dequant_mxfp8(w["wo_a"], w["wo_a_s"]).T)           # B3
    h = bf16_rne(bf16_value(x) + bf16_value(oa) @ dequant_mxfp8(w["wo_b"], w["wo_b_s"]).T)  # B4
    res = dict(xn=xn, qkv=qkv, q_latn=q_latn, kvn=kvn, q=q, o=o, oa=oa, h=h, cache=cache)
    res.update(moe_half(spec, w, x, pos, h))
    return res


def moe_half(spec: dict, w: dict, x, pos, h) -> dict:
    """B5-B10 from the residual h (bf16 bits [R, H])."""
    H, E, K, I = spec["hidden"], spec["n_experts"], spec["topk"], spec["moe_inter"]
    Is, eps, clamp = spec["shared_inter"], spec["eps"], float(spec["swiglu_clamp"])
    R = h.shape[0]
    u = rmsnorm_bits(h, w["ffn_norm"], eps)                                           # B5
    uf = bf16_value(u)
    logits = (uf @ np.asarray(w["router"], np.float32).astype(np.float64).T).astype(np.float32)  # B6
    idx = np.full((R, K), -1, np.int32)
    wts = np.zeros((R, K))
    probs = np.zeros((R, E))
    for r in range(R):
        o_, w_, p_ = topk_route(logits[r], K, float(spec["routed_scale"]))
        probs[r] = p_
        if pos[r] >= 0:
            idx[r], wts[r] = o_, w_
    a = uf @ dequant_mxfp8(w["sh_gu"], w["sh_gu_s"]).T                                # B8
    t_s = bf16_rne(swiglu_clamped(a[:, :Is], a[:, Is:], clamp))
    y_s = bf16_value(t_s) @ dequant_mxfp8(w["sh_d"], w["sh_d_s"]).T
    y_r = np.zeros((R, H))                                                            # B9
    t_r = np.zeros((R, K, I), np.uint16)
    experts = {}
    for r in range(R):
        for j in range(K):
            e = int(idx[r, j])
            if e < 0:
                continue
            if e not in experts:
                experts[e] = (dequant_mxfp4(w["ex_gu"][e], w["ex_gu_s"][e]),
                              dequant_mxfp4(w["ex_d"][e], w["ex_d_s"][e]))
            gu, dn = experts[e]
            ae = gu @ uf[r]
            t = bf16_rne(swiglu_clamped(ae[:I], ae[I:], clamp))
            t_r[r, j] = t
            y_r[r] += wts[r, j] * (dn @ bf16_value(t))
    out = bf16_rne(bf16_value(h) + y_s + y_r)                                         # B10
    pad = np.asarray(pos) < 0
    out[pad] = np.asarray(x, np.uint16)[pad]
    return dict(u=u, logits=logits, probs=probs, topk_idx=idx, topk_w=wts, t_s=t_s, y_s=y_s,
                t_r=t_r, y_r=y_r, out=out)
