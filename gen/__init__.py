"""Seeded synthetic inputs for the fused MoE decode layer.

This module only draws random numbers and packs them into the storage formats the
layer reads: MXFP8 (e4m3 codes + 32x32 E8M0 scales), MXFP4 (packed e2m1 codes + 1x32
E8M0 scales), f32 router weights, bf16 norm gammas and hidden rows, positions, block
tables and a paged fp8 KV cache.  It holds none of the layer's arithmetic: it never
normalises, multiplies weights with activations, attends, routes or quantises a KV
vector the way the layer's insert stage does.  Cached KV records are written from
randomly drawn e4m3 codes and randomly drawn positive per-token scales.

Both the CUDA path (through the product's binding) and the CPU oracle consume what
this module makes; neither side imports the other.

Workloads (dims follow the fused small-batch decode layer of a DeepSeek-style MoE
model; the pages describe MXFP8 attention/shared weights with 32x32 E8M0 scales and
MXFP4 routed experts with 1x32 scales):

* ``tiny``        hidden 256, 4 q heads x 64, one KV latent of 64, q/o ranks 128, window
                  16 over 32 cached tokens in 16-token pages, 8 experts top-2,
                  intermediate 128, 1 row.
* ``small_r11``   a mid-size case spanning several kernel tiles with ragged edges:
                  11 rows over 3 requests (one pad row).
* ``full_r1``     hidden 4096, 64 q heads x 128, KV latent 512, causal window 128,
                  context 8192 in 128-token pages, 128 experts top-6, moe 1024,
                  shared 2048, 1 row.
* ``draft_r6``    as full but top-3, non-causal rows 192 wide, context 65536, the
                  same hidden vector repeated to 6 rows.
* ``full_r48``    as full, 8 requests x 6 rows, contexts uniform in [1024, 65536].
* ``draft_r48``   the draft shape with one request of 48 identical rows: every row routes
                  to the same 3 experts.
"""
from __future__ import annotations

import numpy as np
import torch

# --------------------------------------------------------------------------------------
# Layer dimensions.  q_rank / o_rank are not given on the pages; 1024 makes one full
# layer weigh about 0.9 GB, which is the per-layer size the workloads quote.
# --------------------------------------------------------------------------------------
_TINY = dict(hidden=256, n_q_heads=4, head_dim=64, kv_dim=64, q_rank=128, o_rank=128,
             n_experts=8, topk=2, moe_inter=128, shared_inter=128,
             window=16, swa_width=16, causal=1, block_size=16, kv_record_bytes=80,
             eps=1e-6, swiglu_clamp=7.0, routed_scale=1.0)
_SMALL = dict(hidden=512, n_q_heads=8, head_dim=64, kv_dim=128, q_rank=128, o_rank=128,
              n_experts=16, topk=4, moe_inter=128, shared_inter=256,
              window=24, swa_width=24, causal=1, block_size=16, kv_record_bytes=144,
              eps=1e-6, swiglu_clamp=7.0, routed_scale=1.0)
_FULL = dict(hidden=4096, n_q_heads=64, head_dim=128, kv_dim=512, q_rank=1024, o_rank=1024,
             n_experts=128, topk=6, moe_inter=1024, shared_inter=2048,
             window=128, swa_width=128, causal=1, block_size=128, kv_record_bytes=528,
             eps=1e-6, swiglu_clamp=7.0, routed_scale=1.0)

WORKLOADS = {
    "tiny": dict(spec=_TINY, contexts=[32], rows_per_req=1, pad_rows=0, seed=0),
    "small_r11": dict(spec=_SMALL, contexts=[40, 17, 300], rows_per_req=[4, 3, 3],
                      pad_rows=1, seed=5),
    "full_r1": dict(spec=_FULL, contexts=[8192], rows_per_req=1, pad_rows=0, seed=1),
    "draft_r6": dict(spec=dict(_FULL, topk=3, causal=0, swa_width=192), contexts=[65536],
                     rows_per_req=6, pad_rows=0, seed=2, repeat_input=True),
    "full_r48": dict(spec=_FULL, contexts="uniform:1024:65536:8", rows_per_req=6,
                     pad_rows=0, seed=3),
    # every row identical in one non-causal request: all 48 rows route to the same 3
    # experts (48 routed rows per expert, the most concentrated routing a step can have)
    "draft_r48": dict(spec=dict(_FULL, topk=3, causal=0, swa_width=192), contexts=[40000],
                      rows_per_req=48, pad_rows=0, seed=15, repeat_input=True),
    # parity-only shapes that reach the remaining code paths: 4 one-token requests (a small
    # step whose many expert items do not split K), 24 rows (the 4-tile dense variant), and a
    # narrow layer with 256 experts, top-8, head_dim 64 and a 300-token window (3 splits)
    "full_r4": dict(spec=_FULL, contexts=[3000, 70, 20000, 129], rows_per_req=1, pad_rows=0,
                    seed=11),
    "full_r24": dict(spec=_FULL, contexts="uniform:1024:65536:4", rows_per_req=6, pad_rows=0,
                     seed=12),
    "wide_r9": dict(spec=dict(hidden=1024, n_q_heads=16, head_dim=64, kv_dim=128, q_rank=256,
                              o_rank=256, n_experts=256, topk=8, moe_inter=256,
                              shared_inter=512, window=300, swa_width=300, causal=1,
                              block_size=64, kv_record_bytes=144, eps=1e-6, swiglu_clamp=7.0,
                              routed_scale=2.5),
                    contexts=[400, 350, 900], rows_per_req=[3, 3, 2], pad_rows=1, seed=13),
    # the smallest shapes of the FP4 tensor-core expert path (hidden and intermediate whole
    # 512-element runs, more than 24 routed slots): 13 rows over 3 requests with a pad row,
    # 64 experts top-8 (1 to a few rows per expert); and 20 identical rows top-4, which
    # puts 20 rows on each of 4 experts (a full 16-row group and a ragged 4-row one)
    "mid_r13": dict(spec=dict(hidden=1024, n_q_heads=16, head_dim=64, kv_dim=128, q_rank=256,
                              o_rank=256, n_experts=64, topk=8, moe_inter=512,
                              shared_inter=512, window=64, swa_width=64, causal=1,
                              block_size=64, kv_record_bytes=144, eps=1e-6, swiglu_clamp=7.0,
                              routed_scale=1.5),
                    contexts=[200, 90, 500], rows_per_req=[5, 4, 3], pad_rows=1, seed=16),
    "skew_r20": dict(spec=dict(hidden=1024, n_q_heads=16, head_dim=64, kv_dim=128, q_rank=256,
                               o_rank=256, n_experts=32, topk=4, moe_inter=512,
                               shared_inter=512, window=64, swa_width=64, causal=1,
                               block_size=64, kv_record_bytes=144, eps=1e-6, swiglu_clamp=7.0,
                               routed_scale=1.0),
                     contexts=[300], rows_per_req=20, pad_rows=0, seed=17, repeat_input=True),
}


def spec_of(name: str, **overrides) -> dict:
    s = dict(WORKLOADS[name]["spec"])
    s.update(overrides)
    return s


# --------------------------------------------------------------------------------------
# Storage-format packing used to make weights.  The layer never quantises weights (they
# arrive quantised); this is input preparation only.
# --------------------------------------------------------------------------------------
_E2M1_GRID = torch.tensor([0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0])


def _block_exponent(amax: torch.Tensor, emax_elem: int) -> torch.Tensor:
    """Shared block exponent floor(log2 amax) - emax_elem, kept inside E8M0 codes 1..254."""
    _, e = torch.frexp(amax.clamp_min(1e-30))  # amax = m * 2^e, m in [0.5, 1)
    x = (e - 1) - emax_elem
    return x.clamp(-126, 127)


def pack_mxfp8(w: torch.Tensor):
    """[N, K] float -> (codes u8 [N, K], scales u8 [N/32, K/32]) with 32x32 blocks."""
    n, k = w.shape
    assert n % 32 == 0 and k % 32 == 0
    blk = w.reshape(n // 32, 32, k // 32, 32)
    amax = blk.abs().amax(dim=(1, 3))
    x = _block_exponent(amax, 8)
    scaled = blk / torch.ldexp(torch.ones_like(amax), x.to(amax.dtype))[:, None, :, None]
    codes = scaled.clamp(-448.0, 448.0).to(torch.float8_e4m3fn).view(torch.uint8)
    return codes.reshape(n, k).contiguous(), (x + 127).to(torch.uint8).contiguous()


def pack_mxfp4(w: torch.Tensor):
    """[..., N, K] float -> (packed u8 [..., N, K/2], scales u8 [..., N, K/32]).

    Element 2i sits in the low nibble of byte i, element 2i+1 in the high nibble."""
    *lead, n, k = w.shape
    assert k % 32 == 0
    blk = w.reshape(*lead, n, k // 32, 32)
    amax = blk.abs().amax(dim=-1)
    x = _block_exponent(amax, 2)
    a = (blk / torch.ldexp(torch.ones_like(amax), x.to(amax.dtype))[..., None]).clamp(-6.0, 6.0)
    mag = a.abs()
    # round half to even on the e2m1 grid (steps 0.5 below 2, 1 below 4, 2 above)
    q = torch.where(mag < 2.0, torch.round(mag * 2.0) / 2.0,
                    torch.where(mag < 4.0, torch.round(mag), torch.round(mag / 2.0) * 2.0))
    grid = _E2M1_GRID.to(q.device)
    idx = torch.searchsorted(grid, q.contiguous())
    nib = (idx | ((a < 0) & (idx > 0)).to(idx.dtype) * 8).to(torch.uint8).reshape(*lead, n, k)
    packed = (nib[..., 0::2] | (nib[..., 1::2] << 4)).contiguous()
    return packed, (x + 127).to(torch.uint8).contiguous()


# --------------------------------------------------------------------------------------
# Weights
# --------------------------------------------------------------------------------------
def _gen(seed: int, device) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    return g


def _normal(shape, std, g, device):
    return torch.randn(shape, generator=g, device=device, dtype=torch.float32) * std


def _gamma(n, g, device):
    return (1.0 + 0.1 * torch.randn(n, generator=g, device=device)).to(torch.bfloat16)


def make_weights(spec: dict, seed: int, device="cpu", std: float = 0.02) -> dict:
    """All weights of one layer, seeded.  Matrices are row-major [out, in]."""
    d = torch.device(device)
    g = _gen(seed * 7919 + 17, d)
    H, nq, dh, kv = spec["hidden"], spec["n_q_heads"], spec["head_dim"], spec["kv_dim"]
    qr, orank = spec["q_rank"], spec["o_rank"]
    E, I, Is = spec["n_experts"], spec["moe_inter"], spec["shared_inter"]
    w = {}
    w["attn_norm"] = _gamma(H, g, d)
    w["q_norm"] = _gamma(qr, g, d)
    w["kv_norm"] = _gamma(kv, g, d)
    w["ffn_norm"] = _gamma(H, g, d)
    for name, (n, k) in dict(wqkv=(qr + kv, H), wq_b=(nq * dh, qr), wo_a=(orank, nq * dh),
                             wo_b=(H, orank), sh_gu=(2 * Is, H), sh_d=(H, Is)).items():
        c, s = pack_mxfp8(_normal((n, k), std, g, d))
        w[name], w[name + "_s"] = c, s
    w["router"] = _normal((E, H), std, g, d).contiguous()
    gu_c, gu_s, dn_c, dn_s = [], [], [], []
    for e in range(E):  # one expert at a time keeps the f32 temporaries small
        c, s = pack_mxfp4(_normal((2 * I, H), std, g, d))
        gu_c.append(c), gu_s.append(s)
        c, s = pack_mxfp4(_normal((H, I), std, g, d))
        dn_c.append(c), dn_s.append(s)
    w["ex_gu"], w["ex_gu_s"] = torch.stack(gu_c), torch.stack(gu_s)
    w["ex_d"], w["ex_d_s"] = torch.stack(dn_c), torch.stack(dn_s)
    return w


WEIGHT_KEYS = ["attn_norm", "q_norm", "kv_norm", "ffn_norm", "wqkv", "wqkv_s", "wq_b", "wq_b_s",
               "wo_a", "wo_a_s", "wo_b", "wo_b_s", "router", "sh_gu", "sh_gu_s", "sh_d", "sh_d_s",
               "ex_gu", "ex_gu_s", "ex_d", "ex_d_s"]


# --------------------------------------------------------------------------------------
# Step inputs: hidden rows, positions, request map, block table, paged KV cache
# --------------------------------------------------------------------------------------
def _contexts(desc, rng: np.random.Generator):
    if isinstance(desc, str) and desc.startswith("uniform:"):
        _, lo, hi, n = desc.split(":")
        return [int(v) for v in rng.integers(int(lo), int(hi) + 1, size=int(n))]
    return list(desc)


def make_step(spec: dict, workload: dict, seed: int | None = None, device="cpu",
              prefill_tokens: int | None = None) -> dict:
    """Hidden rows and a paged KV cache for one decode step.

    Request q has ``contexts[q]`` tokens already cached (positions 0..c-1) and
    contributes ``rows_per_req[q]`` new rows at positions c, c+1, ...  Physical pages are
    a random permutation, so every lookup goes through the block table.  Only the last
    ``prefill_tokens`` cached positions of each request (default: the attention reach)
    get random records; the rest stay zero and are never read by a windowed step.
    """
    seed = workload["seed"] if seed is None else seed
    rng = np.random.default_rng(seed + 1000)
    ctx = _contexts(workload["contexts"], rng)
    rpr = workload["rows_per_req"]
    rpr = [rpr] * len(ctx) if isinstance(rpr, int) else list(rpr)
    bs, rec, kvd = spec["block_size"], spec["kv_record_bytes"], spec["kv_dim"]
    reach = max(spec["window"], spec["swa_width"]) + max(rpr) + 8
    prefill = reach if prefill_tokens is None else prefill_tokens

    positions, row_req = [], []
    for q, (c, n) in enumerate(zip(ctx, rpr)):
        positions += [c + i for i in range(n)]
        row_req += [q] * n
    for _ in range(workload.get("pad_rows", 0)):  # pad rows carry position -1
        positions.append(-1)
        row_req.append(0)
    rows = len(positions)

    blocks_per_req = [(c + n + bs - 1) // bs for c, n in zip(ctx, rpr)]
    max_blocks = max(blocks_per_req)
    n_blocks = sum(blocks_per_req) + 3  # a few spare pages that nothing points to
    perm = rng.permutation(n_blocks)
    table = np.zeros((len(ctx), max_blocks), dtype=np.int32)
    o = 0
    for q, nb in enumerate(blocks_per_req):
        table[q, :nb] = perm[o:o + nb]
        o += nb

    cache = np.zeros((n_blocks, bs, rec), dtype=np.uint8)
    for q, c in enumerate(ctx):
        lo = max(0, c - prefill)
        n = c - lo
        if n <= 0:
            continue
        # random e4m3 codes (no NaN) and random positive per-token scales
        vals = rng.standard_normal((n, kvd)).astype(np.float32) * 64.0
        codes = torch.from_numpy(np.clip(vals, -448, 448)).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
        scales = (np.exp2(rng.uniform(-9.0, -5.0, size=n))).astype(np.float32)
        for i, t in enumerate(range(lo, c)):
            blk = table[q, t // bs]
            cache[blk, t % bs, :kvd] = codes[i]
            cache[blk, t % bs, kvd:kvd + 4] = np.frombuffer(scales[i:i + 1].tobytes(), np.uint8)

    g = _gen(seed * 104729 + 3, torch.device("cpu"))
    H = spec["hidden"]
    if workload.get("repeat_input"):
        x = torch.randn((1, H), generator=g).repeat(rows, 1)
    else:
        x = torch.randn((rows, H), generator=g)
    d = torch.device(device)
    return dict(
        rows=rows, contexts=ctx, rows_per_req=rpr,
        x=x.to(torch.bfloat16).to(d),
        positions=torch.tensor(positions, dtype=torch.int32, device=d),
        row_req=torch.tensor(row_req, dtype=torch.int32, device=d),
        block_table=torch.from_numpy(table).to(d),
        kv_cache=torch.from_numpy(cache).to(d),
    )


def make_workload(name: str, device="cpu", seed: int | None = None, weight_device=None,
                  **spec_overrides):
    """(spec, weights, step) for a named workload."""
    wl = WORKLOADS[name]
    spec = spec_of(name, **spec_overrides)
    s = wl["seed"] if seed is None else seed
    weights = make_weights(spec, s, device=weight_device or device)
    step = make_step(spec, wl, seed=s, device=device)
    spec["max_rows"] = max(step["rows"], 1)
    return spec, weights, step


def make_attn_out(spec: dict, step: dict, seed: int = 0, std: float = 0.5, device=None):
    """The attention block's output for every row of a step, as the FFN launch takes it
    (bf16 [rows, H]): an independent normal draw of standard deviation ``std``, on the
    step's device unless ``device`` is given."""
    rows, H = step["rows"], spec["hidden"]
    g = _gen(seed * 7919 + 17, torch.device("cpu"))
    a = torch.randn((rows, H), generator=g) * std
    return a.to(torch.bfloat16).to(device or step["x"].device)


def weight_bytes(spec: dict) -> dict:
    """Bytes of each weight group of one layer, as stored."""
    H, nq, dh, kv = spec["hidden"], spec["n_q_heads"], spec["head_dim"], spec["kv_dim"]
    qr, orank = spec["q_rank"], spec["o_rank"]
    E, I, Is = spec["n_experts"], spec["moe_inter"], spec["shared_inter"]

    def fp8(n, k):
        return n * k + (n // 32) * (k // 32)

    def fp4(n, k):
        return n * k // 2 + n * (k // 32)

    attn = fp8(qr + kv, H) + fp8(nq * dh, qr) + fp8(orank, nq * dh) + fp8(H, orank)
    shared = fp8(2 * Is, H) + fp8(H, Is)
    norms = 2 * (2 * H + qr + kv)
    return dict(attn=attn, shared=shared, router=4 * E * H, norms=norms,
                expert=fp4(2 * I, H) + fp4(H, I))


__all__ = ["WORKLOADS", "spec_of", "make_weights", "make_step", "make_workload", "pack_mxfp8",
           "pack_mxfp4", "weight_bytes", "WEIGHT_KEYS", "make_attn_out"]
