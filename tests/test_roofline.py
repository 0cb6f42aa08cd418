"""The byte / FLOP convention of the bench, pinned to the FLAT blog's printed
forward bandwidths (tests/golden/flat_forward_bandwidth.txt)."""
import os

from chunked_gated_linear_chunk_gb300 import roofline as rf

GOLD = os.path.join(os.path.dirname(__file__), "golden", "flat_forward_bandwidth.txt")


def test_byte_convention_reproduces_flat_forward_bandwidths():
    gate = {"linear_attention": "none", "mamba2": "head", "gla": "channel"}
    for line in open(GOLD):
        if line.startswith("#") or not line.strip():
            continue
        kind, us, tbps = line.split()
        s = rf.Shape(B=8, T=4096, H=16, Hqk=16, K=128, V=128, gate=gate[kind], n_docs=8, final_state=True)
        got = rf.fwd_bytes(s) / (float(us) * 1e-6) / 1e12
        assert abs(got - float(tbps)) < 0.006, (kind, got, tbps)


def test_config2_totals():
    s = rf.Shape(B=4, T=2048, H=16, Hqk=16, K=128, V=128)
    assert abs(rf.fwd_flops(s) / 1e9 - 12.88) < 0.01
    assert abs(rf.bwd_flops(s) / 1e9 - 32.21) < 0.01
    assert abs(rf.fwd_bytes(s) / 1e6 - 201.3) < 0.1
    assert abs(rf.bwd_bytes(s) / 1e6 - 369.1) < 0.1
    t = rf.roofline_time_s(rf.fwd_flops(s) + rf.bwd_flops(s), rf.fwd_bytes(s) + rf.bwd_bytes(s), 1956.5, 6680.8)
    assert abs(t * 1e6 - 85.4) < 0.1


def test_per_kernel_bytes_add_up():
    s = rf.Shape(B=4, T=2048, H=16, Hqk=16, K=128, V=128)
    ins5 = rf.kernel_bytes(s, "gla_bwd_dq_kernel") - s.qk_bytes()
    assert ins5 == rf.bwd_bytes(s) - (2 * s.qk_bytes() + s.v_bytes() + s.gate_bytes())
    outs = (rf.kernel_bytes(s, "gla_bwd_dq_kernel") - ins5) + (rf.kernel_bytes(s, "gla_bwd_rev_kernel") - ins5)
    assert outs == 2 * s.qk_bytes() + s.v_bytes() + s.gate_bytes()
