"""Algorithmic bytes and FLOPs of the path (measurement convention).

Bytes follow the convention the FLAT blog uses for its bandwidth figures
(trainstation-project.github.io/blog/flat, "Benchmark Setup" and the
forward "Throughput" paragraph): every input read once and every output
written once per call, the final state in fp32.  Chunk states, re-reads
and workspace traffic are not counted; they count against the kernel.

FLOPs: matmul FLOPs of the chunk form at chunk length C with full
(unmasked) C x C blocks, per token (q/k terms once per q/k head):
    forward   Hqk * 2CK + H * (2CV + 4KV)
    backward  Hqk * 6CK + H * (4CV + 10KV)
(QK^T, PV, readout, state update; backward adds the recomputed QK^T,
the dq/dk intra products, dP, the dv intra product and five state-sized
products).  Exponentials and masks are not counted.
"""
from __future__ import annotations

from dataclasses import dataclass


@dataclass(frozen=True)
class Shape:
    B: int
    T: int
    H: int
    Hqk: int
    K: int
    V: int
    elem: int = 2  # bytes per q/k/v/o element
    gate: str = "channel"  # "channel" (GLA, fp32 [B,T,H,K]), "head" (SSD, [B,T,H]) or "none"
    n_docs: int = 0
    initial_state: bool = False
    final_state: bool = False
    dht: bool = False
    chunk: int = 64
    plen: int = 0  # piece length of the backward's exact sequence split (0: no split)

    @property
    def BT(self):
        return self.B * self.T

    def gate_bytes(self):
        if self.gate == "channel":
            return self.BT * self.H * self.K * 4
        if self.gate == "head":
            return self.BT * self.H * 4
        return 0

    def qk_bytes(self):
        return self.BT * self.Hqk * self.K * self.elem

    def v_bytes(self):
        return self.BT * self.H * self.V * self.elem

    def state_bytes(self):
        return self.n_docs * self.H * self.K * self.V * 4


def fwd_bytes(s: Shape) -> int:
    b = 2 * s.qk_bytes() + s.v_bytes() + s.gate_bytes() + s.v_bytes()  # q, k, v, g in; o out
    if s.initial_state:
        b += s.state_bytes()
    if s.final_state:
        b += s.state_bytes()
    return b


def bwd_bytes(s: Shape) -> int:
    b = 2 * s.qk_bytes() + 2 * s.v_bytes() + s.gate_bytes()  # q, k, v, g, do in
    b += 2 * s.qk_bytes() + s.v_bytes() + s.gate_bytes()  # dq, dk, dv, dg out
    if s.initial_state:
        b += 2 * s.state_bytes()  # h0 in, dh0 out
    if s.dht:
        b += s.state_bytes()
    return b


def fwd_flops(s: Shape) -> int:
    C, K, V = s.chunk, s.K, s.V
    return s.BT * (s.Hqk * 2 * C * K + s.H * (2 * C * V + 4 * K * V))


def bwd_flops(s: Shape) -> int:
    C, K, V = s.chunk, s.K, s.V
    return s.BT * (s.Hqk * 6 * C * K + s.H * (4 * C * V + 10 * K * V))


def kernel_bytes(s: Shape, label: str) -> int:
    """Algorithmic bytes of one launch of the named kernel: the inputs it
    must read and the outputs it must write (each once)."""
    ins5 = 2 * s.qk_bytes() + 2 * s.v_bytes() + s.gate_bytes()
    if label in ("gla_fwd_kernel", "simt_fwd", "ssd_fwd_kernel"):
        return fwd_bytes(s)
    if label in ("gla_bwd_dq_kernel", "ssd_bwd_a_kernel"):  # reads q, k, v, g, do (+h0, dht); writes dq
        return ins5 + s.qk_bytes() + (s.state_bytes() if s.initial_state else 0) + (
            s.state_bytes() if s.dht else 0)
    if label in ("gla_bwd_rev_kernel", "ssd_bwd_b_kernel"):  # reads q, k, v, g, do (+dht); writes dk, dv, dg (+dh0)
        return ins5 + s.qk_bytes() + s.v_bytes() + s.gate_bytes() + (
            s.state_bytes() if s.dht else 0) + (s.state_bytes() if s.initial_state else 0)
    if label == "piece_state_kernel" and s.plen > 0:
        # the forward piece pass reads k, v, g of every piece but a row's
        # last, the reverse pass q, do, g of every piece but its first
        npr = -(-s.T // s.plen)
        per_tok = s.Hqk * s.K * s.elem + s.H * s.V * s.elem + s.gate_bytes() // s.BT
        return s.B * ((npr - 1) * s.plen + (s.T - s.plen)) * per_tok
    if label == "simt_state_pass":  # reads k, v, g (+h0)
        return s.qk_bytes() + s.v_bytes() + s.gate_bytes() + (s.state_bytes() if s.initial_state else 0)
    if label == "simt_bwd":
        return bwd_bytes(s)
    return 0


def piece_len(B: int, T: int, n_seqs: int, H: int, sms: int, chunk: int = 64) -> int:
    """The backward's piece length for uniform rows (0: no split), by the
    library's rule: split only when one CTA per (document, head) leaves more
    than a quarter of the SMs idle, into about as many pieces as fill one
    wave, each a whole number of chunks and at least four."""
    units = n_seqs * H
    if units <= 0 or units * 4 >= sms * 3:
        return 0
    want = sms // units
    if want < 2:
        return 0
    avg = -(-(B * T) // n_seqs)
    plen = -(-avg // want)
    plen = max(-(-plen // chunk) * chunk, 4 * chunk)
    return 0 if plen >= avg else plen


def roofline_time_s(flops: float, nbytes: float, peak_tflops: float, peak_gbs: float) -> float:
    return max(flops / (peak_tflops * 1e12), nbytes / (peak_gbs * 1e9))
