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


def test_piece_length_rule():
    # one CTA per (document, head) in the backward: split only when that
    # leaves more than a quarter of 152 SMs idle, into about one wave
    assert rf.piece_len(4, 2048, 4, 16, 152) == 1024  # 64 units -> two pieces per row
    assert rf.piece_len(1, 65536, 1, 16, 152) == 7296  # 16 units -> nine pieces per row
    assert rf.piece_len(4, 4096, 4, 32, 152) == 0  # 128 units fill the GPU
    assert rf.piece_len(1, 300, 1, 16, 152) == 256  # at least four chunks per piece
    assert rf.piece_len(1, 200, 1, 16, 152) == 0  # a piece would not be shorter than the row


def test_piece_pass_bytes_match_an_explicit_walk_over_the_pieces():
    for (B, T, H, plen) in ((4, 2048, 16, 1024), (1, 65536, 16, 7296), (2, 1000, 3, 256)):
        s = rf.Shape(B=B, T=T, H=H, Hqk=H, K=128, V=128, plen=plen)
        starts = list(range(0, T, plen))
        fwd_tok = sum(min(T, p + plen) - p for p in starts[:-1])  # every piece but a row's last
        rev_tok = sum(min(T, p + plen) - p for p in starts[1:])  # every piece but a row's first
        per_tok_fwd = H * 128 * 2 + H * 128 * 2 + H * 128 * 4  # k, v bf16 and g fp32 per token
        per_tok_rev = H * 128 * 2 + H * 128 * 2 + H * 128 * 4  # q, do bf16 and g fp32 per token
        want = B * (fwd_tok * per_tok_fwd + rev_tok * per_tok_rev)
        assert rf.kernel_bytes(s, "piece_state_kernel") == want, (B, T, H, plen)
    # workload 2: the bytes the ncu capture of the piece pass reads (134.3 MB)
    s = rf.Shape(B=4, T=2048, H=16, Hqk=16, K=128, V=128, plen=1024)
    assert rf.kernel_bytes(s, "piece_state_kernel") == 134217728
    assert rf.kernel_bytes(rf.Shape(B=4, T=2048, H=16, Hqk=16, K=128, V=128), "piece_state_kernel") == 0
