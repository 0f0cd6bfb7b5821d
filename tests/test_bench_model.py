"""The byte and flop counts behind bench.py's roofline fractions (CPU only).

The ZeCO operator's algorithmic work per token and head is fixed by the
method's passes: the forward reads k, v, g in pass 1 and q, k, v, g in pass 2
and writes o; the backward's pre-pass reads q, do, g and its main pass reads
q, k, v, g, do and writes dq, dk, dv, dg; the segment states add 16 d_k d_v
bytes (forward) and 20 d_k d_v bytes (backward) per segment.  These tests pin
bench.py's formulas to those counts at the 1M-token workload (d_k = 256,
d_v = 512, L = 16,384, bf16)."""
import bench

DK, DV, L, C = 256, 512, 16384, 64


def test_operator_bytes_and_flops_per_token_head():
    fwd = bench.zeco_operator_bytes_per_token(DK, DV, L, bwd=False)
    assert fwd == 2 * (5 * DK + 3 * DV) + 16 * DK * DV / L == 5632 + 128
    both = bench.zeco_operator_bytes_per_token(DK, DV, L)
    assert both == 5632 + 8192 + 36 * DK * DV / L == 14112
    assert bench.zeco_operator_flops_per_token(DK, DV, C, bwd=False) == 884736
    assert bench.zeco_operator_flops_per_token(DK, DV, C) == 884736 + 1802240


def test_step_roofline_at_the_headline_workload():
    tokens_heads = 4 * (1 << 20)
    nbytes = bench.zeco_operator_bytes_per_token(DK, DV, L) * tokens_heads
    assert abs(nbytes / 1e9 - 59.19) < 0.01
    assert abs(nbytes / 6752.4e9 * 1e3 - 8.766) < 0.001  # ms at the measured HBM copy rate


def test_method_bytes_count_each_input_and_output_once():
    m = bench.method_bytes_per_token(DK, DV, L)
    st = DK * DV * 4 / L
    # pass 1 reads k, g, v; pass 2 reads q, k, g, v and writes o; the decay pass reads
    # q, k, g (its outputs are intermediates), the score passes only intermediates
    assert m["chunk_state"] == 2 * (2 * DK + DV) + st
    assert m["fwd_out"] == 2 * (3 * DK + 2 * DV) + st
    assert m["A"] == 0.0
    # dk sweep: q, k, g, v, do and its state in, dk and dg out
    assert m["bwd_dk"] == 2 * (3 * DK + 2 * DV) + 2 * 2 * DK + st


def test_implementation_bytes_of_the_tensor_core_step():
    kb = bench.kernel_bytes_per_token(DK, DV, L)
    tc = ("decay", "A", "chunk_state", "seg_scan_fwd", "fwd_out", "dA", "dstate_local",
          "seg_scan_rev", "bwd_dv", "bwd_dq", "bwd_dk")
    total = sum(kb[k] for k in tc)
    assert total == 26832
    assert abs(total / bench.zeco_operator_bytes_per_token(DK, DV, L) - 1.9014) < 1e-4


def test_scan_overlap_instrument_on_synthetic_intervals():
    # the pages' Eq. 11 instrument: the share of the scan's kernel time during which
    # no diagonal-attention kernel (A forward, dA backward) runs
    iv = [("tc_A", 0.0, 1.0), ("seg_scan_fwd", 0.5, 1.5),      # half of the scan overlapped
          ("tc_dA", 2.0, 3.0), ("seg_scan_rev", 2.0, 2.5)]     # all of it overlapped
    out = bench.scan_overlap(iv)
    assert abs(out["fwd"]["non_overlapped_frac"] - 0.5) < 1e-12
    assert abs(out["bwd"]["non_overlapped_frac"] - 0.0) < 1e-12
    assert abs(out["fwd"]["scan_ms"] - 1.0) < 1e-12
    # no diagonal-attention kernel in the run: no figure for that direction
    assert "fwd" not in bench.scan_overlap([("seg_scan_fwd", 0.0, 1.0)])


def test_kernel_names_map_to_their_byte_counts():
    kb = bench.kernel_bytes_per_token(DK, DV, L)
    for name in ("tc_decay", "tc_A", "tc_chunk_state", "seg_scan_fwd", "tc_fwd_out", "tc_dA",
                 "tc_dstate_local", "seg_scan_rev", "tc_bwd_dv", "tc_bwd_dq", "tc_bwd_dk"):
        assert bench.canonical_kernel(name) in kb, name
    assert bench.canonical_kernel("tc_dA") == "dA" and bench.canonical_kernel("tc_A") == "A"
