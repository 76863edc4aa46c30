"""The algorithmic byte counts behind the bench's GB/s and roofline figures.

Each weight group's byte count is checked against the bytes of the tensors the generator
actually builds, for the tiny and the mid-size layer, so the formula cannot drift from the
storage format. The full-size layer (hidden 4096, 128 experts of 1024, shared 2048) must
come to about 0.9 GB, nearly all of it routed-expert weights. One test also ties the
dominant launch's byte count to the 48-row workload's routing.
"""
import pytest

import bench
import gen

GROUPS = {
    "attn": ("wqkv", "wqkv_s", "wq_b", "wq_b_s", "wo_a", "wo_a_s", "wo_b", "wo_b_s"),
    "shared": ("sh_gu", "sh_gu_s", "sh_d", "sh_d_s"),
    "router": ("router",),
    "norms": ("attn_norm", "q_norm", "kv_norm", "ffn_norm"),
}


@pytest.mark.parametrize("name", ["tiny", "small_r11"])
def test_weight_bytes_are_the_generated_tensors_bytes(name):
    spec, w, _ = gen.make_workload(name)
    wb = gen.weight_bytes(spec)
    for group, keys in GROUPS.items():
        assert wb[group] == sum(w[k].nbytes for k in keys), group
    E = spec["n_experts"]
    assert wb["expert"] * E == sum(w[k].nbytes for k in ("ex_gu", "ex_gu_s", "ex_d", "ex_d_s"))
    # the routed GEMMs' weight terms: every expert hit, no activation rows
    assert bench.expert_gate_up_bytes(spec, E, 0, 0) == w["ex_gu"].nbytes + w["ex_gu_s"].nbytes
    assert bench.expert_down_bytes(spec, E, 0) == w["ex_d"].nbytes + w["ex_d_s"].nbytes


def test_routed_launch_bytes_grow_by_one_expert_matrix_per_hit_expert():
    spec, w, _ = gen.make_workload("tiny")
    E = spec["n_experts"]
    gu = (w["ex_gu"].nbytes + w["ex_gu_s"].nbytes) // E
    d = (w["ex_d"].nbytes + w["ex_d_s"].nbytes) // E
    for hit in range(1, E + 1):
        assert bench.expert_gate_up_bytes(spec, hit, 5, 3) - bench.expert_gate_up_bytes(spec, hit - 1, 5, 3) == gu
        assert bench.expert_down_bytes(spec, hit, 5) - bench.expert_down_bytes(spec, hit - 1, 5) == d


def test_full_size_layer_is_about_0_9_gb():
    spec = gen.spec_of("full_r48")
    wb = gen.weight_bytes(spec)
    total = wb["attn"] + wb["shared"] + wb["router"] + wb["norms"] + spec["n_experts"] * wb["expert"]
    assert 0.85e9 < total < 0.95e9, total
    # the experts are the bulk of it: the dominant kernels stream them
    assert spec["n_experts"] * wb["expert"] > 0.9 * total


def test_dominant_launch_bytes_at_the_headline_routing():
    """48 rows x top-6 = 288 routed slots over 111 hit experts (the routing of the 48-row
    workload's first weight copy): one gate_up launch must move every hit expert's gate_up
    matrix and scales, read the 48 normed rows and write the 288 SwiGLU rows."""
    spec = gen.spec_of("full_r48")
    H, I = spec["hidden"], spec["moe_inter"]
    one_expert_gate_up = 2 * I * H // 2 + 2 * I * H // 32  # e2m1 codes + 1x32 E8M0 scales
    assert one_expert_gate_up == 4_456_448
    got = bench.expert_gate_up_bytes(spec, 111, 288, 48)
    assert got == 111 * one_expert_gate_up + 48 * H * 2 + 288 * I * 2 == 495_648_768
