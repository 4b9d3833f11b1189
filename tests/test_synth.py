"""The seeded generator: torch SplitMix64 equals the scalar definition; streams are index-addressed."""
import torch

from moe_expert_ffn_03_gb300 import configs, synth


def test_splitmix64_matches_scalar_definition():
    key = synth.stream_key(0, 3)
    got = synth.raw_u64(key, 10, 5, "cpu").tolist()
    want = []
    for i in range(10, 15):
        state = (key + (i + 1) * 0x9E3779B97F4A7C15) & ((1 << 64) - 1)
        v = synth.splitmix64_py(state)
        want.append(v - (1 << 64) if v >= 1 << 63 else v)
    assert got == want


def test_normal_stream_is_chunk_independent():
    key = synth.stream_key(5, 1)
    a = synth.normal_f64(key, 1000, "cpu")
    b = synth.normal_f64(key, 600, "cpu", start=400)
    assert torch.equal(a[400:], b)
    assert abs(float(a.mean())) < 0.15 and abs(float(a.std()) - 1.0) < 0.1


def test_workload_inputs_shapes_and_routing_structure():
    w = configs.get(0)
    d = synth.make_inputs(w, 0)
    assert d["x"].shape == (w.T, w.H) and d["x"].dtype == torch.bfloat16
    assert d["w_gu"].shape == (w.E, 2 * w.I, w.H) and d["w_d"].shape == (w.E, w.H, w.I)
    assert d["dout"].shape == (w.T, w.H)
    small_zipf = configs.small(2048, 64, 128, 8, 2, routing="zipf", backward=False)
    lz = synth.make_logits(small_zipf, 0, "cpu")
    top1 = lz.argmax(dim=1)
    counts = torch.bincount(top1, minlength=8)
    assert counts[7] == 0 and counts[0] > counts[1] > counts[3]
