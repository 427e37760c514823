"""The seeded input generator: determinism, chain subsets, shapes and dtypes."""
import torch

from test_weight_sequence_ttt_b300.inputs import WORKLOADS, make_inputs


def test_deterministic_and_subset_matches_full():
    w = WORKLOADS["linear_b8h12_d64_t2k"].with_(T=64)
    a = make_inputs(w)
    b = make_inputs(w)
    for k in ("Q", "K", "V", "eta", "W0"):
        assert torch.equal(a[k], b[k])
    sub = make_inputs(w, chains=[5, 30])
    for i, ch in enumerate([5, 30]):
        bi, hi = divmod(ch, w.H)
        for k in ("Q", "K", "V", "eta"):
            assert torch.equal(sub[k][i, 0], a[k][bi, hi])
        assert torch.equal(sub["W0"][i, 0], a["W0"][0, hi])


def test_shapes_dtypes_and_ranges():
    w = WORKLOADS["mlp_b4h12_d64_t8k"].with_(T=32)
    x = make_inputs(w)
    assert x["Q"].shape == (4, 12, 32, 64) and x["Q"].dtype == torch.bfloat16
    assert x["W1"].shape == (1, 12, 256, 64) and x["W2"].shape == (1, 12, 64, 256)
    assert x["eta"].dtype == torch.float32
    assert 0.3 < x["eta"].mean().item() < 0.7 and x["eta"].min() > 0
    t = make_inputs(WORKLOADS["linear_f32_tiny"])
    assert t["Q"].dtype == torch.float32 and t["Q"].shape == (1, 1, 64, 16)


def test_cotangents_shapes_and_subsets():
    from test_weight_sequence_ttt_b300.inputs import make_cotangents
    w = WORKLOADS["linear_b8h12_d64_t2k"].with_(T=32)
    c = make_cotangents(w)
    assert c["dZ"].shape == (8, 12, 32, 64) and c["dZ"].dtype == torch.bfloat16
    assert c["dW_n"].shape == (8, 12, 64, 64) and c["dc_n"].shape == (8, 12, 64)
    sub = make_cotangents(w, chains=[7, 50])
    for i, ch in enumerate([7, 50]):
        bi, hi = divmod(ch, w.H)
        for k in ("dZ", "dW_n", "dc_n"):
            assert torch.equal(sub[k][i, 0], c[k][bi, hi]), k
    m = make_cotangents(WORKLOADS["mlp_b4h12_d64_t8k"].with_(T=16))
    assert m["dW1_n"].shape == (4, 12, 256, 64) and m["dc1_n"].shape == (4, 12, 256)
    assert m["dW2_n"].shape == (4, 12, 64, 256) and m["dc2_n"].shape == (4, 12, 64)
    # distinct streams: the seeds are not copies of one another
    assert not torch.equal(m["dc2_n"], m["dc1_n"][..., :64])
