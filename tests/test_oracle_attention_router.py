"""Pins for the oracle's KV insert, windowed attention and router.

Attention is pinned by closed forms (identical keys give the mean of the values; one
key gives its value; a zero query gives the plain mean of the window's values, which a
numpy loop over the decoded cache computes independently) and by invariances (paging,
records outside the window).  The router is pinned by brute-force sorting.
"""
import copy

import numpy as np
import pytest
import torch

import gen
from tests.helpers import bf16_f64, np_inputs


def _bf16(a):
    return torch.from_numpy(np.asarray(a, np.float32)).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


def _decode_record(rec, kv_dim):
    codes = torch.from_numpy(np.ascontiguousarray(rec[:kv_dim])).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    scale = np.frombuffer(rec[kv_dim:kv_dim + 4].tobytes(), np.float32)[0]
    return codes * float(scale)


def _workload(name="small_r11"):
    spec, w, st = gen.make_workload(name)
    wn, sn = np_inputs(w, st)
    return spec, wn, sn


# ----------------------------------------------------------------------------- attend
def test_attend_identical_keys_give_mean_of_values(orc):
    rng = np.random.default_rng(0)
    k = np.tile(rng.standard_normal(16), (7, 1))
    v = rng.standard_normal((7, 16))
    out = orc.attend(rng.standard_normal(16), k, v, 0.25)
    np.testing.assert_allclose(out, v.mean(0), rtol=1e-13, atol=1e-14)


def test_attend_single_key_and_dominant_key(orc):
    rng = np.random.default_rng(1)
    v = rng.standard_normal((1, 8))
    np.testing.assert_allclose(orc.attend(rng.standard_normal(8), rng.standard_normal((1, 8)), v, 1.0), v[0])
    q = np.zeros(8)
    q[0] = 1.0
    keys = np.zeros((5, 8))
    keys[3, 0] = 1000.0                                  # score 1000 vs 0: weight ~ 1
    vals = rng.standard_normal((5, 8))
    np.testing.assert_allclose(orc.attend(q, keys, vals, 1.0), vals[3], atol=1e-12)


# -------------------------------------------------------------------------- key range
def test_key_range_causal_and_noncausal(orc):
    spec, _, st = _workload()
    W = spec["window"]
    for r, p in enumerate(st["positions"]):
        rng_ = orc.key_range(spec, st, r)
        if p < 0:
            assert rng_ is None
        else:
            assert rng_ == (max(0, p - W + 1), p)
    nc = dict(spec, causal=0, swa_width=20)
    for r, p in enumerate(st["positions"]):
        if p < 0:
            continue
        q = st["row_req"][r]
        e = max(pp for pp, qq in zip(st["positions"], st["row_req"]) if qq == q)
        assert orc.key_range(nc, st, r) == (max(0, e - 20 + 1), e)


# ---------------------------------------------------------------------------- insert
def test_kv_insert_layout_paging_and_pad_rows(orc):
    spec, _, st = _workload()
    R, kvd, bs = len(st["positions"]), spec["kv_dim"], spec["block_size"]
    kvn = _bf16(np.random.default_rng(2).standard_normal((R, kvd)))
    rc, cache = orc.kv_insert(spec, st, kvn)
    assert rc == 0
    before = st["kv_cache"]
    touched = np.zeros(before.shape[:2], bool)
    for r, (p, q) in enumerate(zip(st["positions"], st["row_req"])):
        if p < 0:
            continue
        blk = st["block_table"][q, p // bs]
        rec = cache[blk, p % bs]
        codes, s = orc.kv_quant(kvn[r])
        assert np.array_equal(rec[:kvd], codes)
        assert np.frombuffer(rec[kvd:kvd + 4].tobytes(), np.float32)[0] == s
        assert np.array_equal(rec[kvd + 4:], before[blk, p % bs, kvd + 4:])   # pad bytes kept
        touched[blk, p % bs] = True
    assert np.array_equal(cache[~touched], before[~touched])                 # nothing else moved


def test_kv_insert_refuses_overlapping_pages(orc):
    spec, _, st = _workload()
    bad = dict(st)
    # a [blocks, block, record] view whose block stride is shorter than block * record
    c = st["kv_cache"]
    nb, bs, rec = c.shape
    bad["kv_cache"] = np.zeros((nb, bs - 1, rec), np.uint8)
    kvn = np.zeros((len(st["positions"]), spec["kv_dim"]), np.uint16)
    rc, _ = orc.kv_insert(spec, bad, kvn)
    assert rc == -1


# ------------------------------------------------------------------------- attention
def _window_means(spec, st, cache):
    """Mean of each head's value slice over the row's window, by direct loops."""
    nq, dh, kvd, bs = spec["n_q_heads"], spec["head_dim"], spec["kv_dim"], spec["block_size"]
    G = kvd // dh
    out = np.zeros((len(st["positions"]), nq * dh))
    for r, (p, q) in enumerate(zip(st["positions"], st["row_req"])):
        if p < 0:
            continue
        lo, hi = max(0, p - spec["window"] + 1), p
        vals = np.stack([_decode_record(cache[st["block_table"][q, t // bs], t % bs], kvd)
                         for t in range(lo, hi + 1)])
        for h in range(nq):
            g = h // (nq // G)
            out[r, h * dh:(h + 1) * dh] = vals[:, g * dh:(g + 1) * dh].mean(0)
    return out


def test_attention_zero_query_is_window_mean(orc):
    spec, _, st = _workload()
    R, QW = len(st["positions"]), spec["n_q_heads"] * spec["head_dim"]
    q = np.zeros((R, QW), np.uint16)                    # all scores equal -> uniform weights
    rc, o = orc.attention(spec, st, q)
    assert rc == 0
    want = _window_means(spec, st, st["kv_cache"])
    got = bf16_f64(o)
    np.testing.assert_allclose(got, want, rtol=2.0 ** -8, atol=1e-30)  # bf16 of the exact mean
    assert not got[np.array(st["positions"]) < 0].any() # pad rows give zero


def test_attention_paging_invariance_and_window_locality(orc):
    spec, _, st = _workload()
    R, QW, bs = len(st["positions"]), spec["n_q_heads"] * spec["head_dim"], spec["block_size"]
    q = _bf16(np.random.default_rng(3).standard_normal((R, QW)))
    _, o_ref = orc.attention(spec, st, q)
    # same logical content behind a different page permutation
    perm = np.random.default_rng(4).permutation(st["kv_cache"].shape[0])
    st2 = copy.deepcopy(st)
    st2["kv_cache"] = np.empty_like(st["kv_cache"])
    st2["kv_cache"][perm] = st["kv_cache"]
    st2["block_table"] = perm[st["block_table"]].astype(np.int32)
    _, o2 = orc.attention(spec, st2, q)
    assert np.array_equal(o_ref, o2)
    # a record just outside row 0's window does not matter; one inside does
    p, rq = st["positions"][0], st["row_req"][0]
    lo = p - spec["window"] + 1
    for t, changes in [(lo - 1, False), (lo, True)]:
        st3 = copy.deepcopy(st)
        st3["kv_cache"][st["block_table"][rq, t // bs], t % bs, :spec["kv_dim"]] ^= 0x11
        _, o3 = orc.attention(spec, st3, q)
        assert (not np.array_equal(o3[0], o_ref[0])) == changes


# ---------------------------------------------------------------------------- router
def test_router_matches_brute_force_sort(orc):
    rng = np.random.default_rng(5)
    R, E, H, k = 9, 32, 256, 5
    u = _bf16(rng.standard_normal((R, H)))
    wr = (rng.standard_normal((E, H)) * 0.05).astype(np.float32)
    res = orc.router(u, wr, k, routed_scale=2.5)
    z_ref = (bf16_f64(u) @ wr.astype(np.float64).T)
    np.testing.assert_allclose(res["logits"], z_ref.astype(np.float32), rtol=1e-6, atol=1e-6)
    z = res["logits"].astype(np.float64)
    for r in range(R):
        order = np.argsort(-z[r], kind="stable")[:k]    # stable: ties keep the lower index
        assert list(res["idx"][r]) == list(order)
        p = np.exp(z[r] - z[r].max())
        p /= p.sum()
        np.testing.assert_allclose(res["probs"][r], p, rtol=1e-12)
        np.testing.assert_allclose(res["w"][r], p[order] / p[order].sum() * 2.5, rtol=1e-12)


def test_router_ties_go_to_lower_index_and_pad_rows(orc):
    H, E = 64, 8
    wr = np.zeros((E, H), np.float32)
    wr[[2, 5, 6], 0] = 1.0                               # experts 2, 5, 6 tie
    u = _bf16(np.ones((2, H)))
    res = orc.router(u, wr, 2, positions=np.array([3, -1], np.int32))
    assert list(res["idx"][0]) == [2, 5]
    np.testing.assert_allclose(res["w"][0], [0.5, 0.5])
    assert list(res["idx"][1]) == [-1, -1] and not res["w"][1].any()


def test_router_force_idx(orc):
    rng = np.random.default_rng(6)
    u = _bf16(rng.standard_normal((2, 64)))
    wr = rng.standard_normal((8, 64)).astype(np.float32)
    forced = np.array([[7, 1], [0, 3]], np.int32)
    res = orc.router(u, wr, 2, force_idx=forced)
    assert np.array_equal(res["idx"], forced)
    p = res["probs"]
    for r in range(2):
        np.testing.assert_allclose(res["w"][r], p[r, forced[r]] / p[r, forced[r]].sum())


# ------------------------------------------------------------------ attention scale pin
def test_attention_score_scale_two_key_closed_form(orc):
    """Scaled dot-product attention (softmax(q . k / sqrt(head_dim))) pinned by a closed form.

    One row at position 1 with a causal window of 2 sees two keys.  In latent slice g the
    newer key holds 2 at element 0 and (1 + g/4) at element 1, the older key 0 and -1; head
    h's query is a_h e_0.  The score difference is then 2 a_h / sqrt(64), so the newer key's
    weight is w = 1 / (1 + exp(-2 a_h / 8)) and o_h[0] = 2 w, o_h[1] = (1 + g/4) w - (1 - w).
    Scales 1/sqrt(kv_dim) = 1/16, 1/head_dim and 1 give weights off by far more than a bf16
    rounding, and a wrong head -> slice map changes o_h[1]; both would fail."""
    nq, dh, kvd = 4, 64, 256                       # 4 latent slices, one head each
    rec_bytes = 272
    spec = dict(gen.spec_of("tiny"), n_q_heads=nq, head_dim=dh, kv_dim=kvd, window=2,
                swa_width=2, causal=1, block_size=16, kv_record_bytes=rec_bytes)
    cache = np.zeros((1, 16, rec_bytes), np.uint8)
    one = np.frombuffer(np.float32(1.0).tobytes(), np.uint8)
    e4m3 = {2.0: 0x40, 1.0: 0x38, 1.25: 0x3A, 1.5: 0x3C, 1.75: 0x3E, -1.0: 0xB8}
    for g in range(nq):
        cache[0, 1, g * dh + 0] = e4m3[2.0]
        cache[0, 1, g * dh + 1] = e4m3[1.0 + g / 4]
        cache[0, 0, g * dh + 1] = e4m3[-1.0]
    cache[0, 0, kvd:kvd + 4] = one
    cache[0, 1, kvd:kvd + 4] = one
    a = np.array([4.375, 1.5, -2.0, 0.75])         # exact in bf16
    q = np.zeros(nq * dh)
    q[np.arange(nq) * dh] = a
    st = dict(x=np.zeros((1, spec["hidden"]), np.uint16), positions=np.array([1], np.int32),
              row_req=np.array([0], np.int32), block_table=np.zeros((1, 1), np.int32),
              kv_cache=cache)
    rc, o = orc.attention(spec, st, _bf16(q[None, :]))
    assert rc == 0
    got = bf16_f64(o[0]).reshape(nq, dh)

    def expect(scale):
        w = 1.0 / (1.0 + np.exp(-2.0 * a * scale))
        g = np.arange(nq)
        return np.stack([2 * w, (1 + g / 4) * w - (1 - w)], axis=1)

    want = expect(1.0 / np.sqrt(dh))
    np.testing.assert_allclose(got[:, :2], want, rtol=2.0 ** -8, atol=0)
    assert not got[:, 2:].any()                    # every other element is zero in both keys
    for wrong in (1.0 / np.sqrt(kvd), 1.0 / dh, 1.0):
        assert np.abs(expect(wrong) - want).max() > 8 * 2.0 ** -8 * np.abs(want).max()
