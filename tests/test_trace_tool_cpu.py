"""The tracing build's reader (block_scaled_moe_gb300/trace.py) on synthetic stamps: the summaries
are arithmetic over the stamp arrays, so a hand-built trace with known gaps must come back with
exactly those gaps.  No GPU and no tracing library are needed."""

import numpy as np

from block_scaled_moe_gb300 import trace


def _synthetic_fused_stages(n1=3, n2=4, kt1=5, kt2=3, period=700, enter=100, decode=50, prefetch=80, to_wait=40,
                            mma_decode=300, mma_to_wait=60, bubble=900):
    """A two-CTA stage trace in which every stage follows the previous one by `period` cycles, except
    the first stage of each unit after the first, which comes `bubble` cycles later still; the unit
    stamps sit at fixed offsets from the last stage of the previous unit."""
    st = np.zeros((2, trace.FUSED_STAGE_EVENTS, trace.FUSED_STAGES), np.int64)
    kts = [kt1] * n1 + [kt2] * n2
    starts = np.cumsum([0] + kts[:-1])
    n = int(sum(kts))
    for cta in range(2):
        t = 10_000
        m0 = np.zeros(n, np.int64)
        for i in range(n):
            t += period + (bubble if i in set(starts[1:].tolist()) else 0)
            m0[i] = t
        s = st[cta]
        s[2, :n] = m0                # MMA chain 0 saw the stage full
        s[3, :n] = m0 + 200          # chain 0 issued
        s[1, :n] = m0 - 3000         # producer issued
        s[0, :n] = m0 - 3100         # producer got the slot
        for u in range(1, len(kts)):
            b = starts[u]
            s[12, u] = s[1, b - 1] + enter
            s[13, u] = s[12, u] + decode
            s[14, u] = s[13, u] + prefetch
            s[6, b] = s[14, u] + to_wait
            s[15, u] = s[3, b - 1] + mma_decode
            s[10, b] = s[15, u] + mma_to_wait
    return st


def test_transition_costs_recover_the_planted_gaps():
    st = _synthetic_fused_stages()
    c = trace.transition_costs(st, 0, 3, 7, 5, 3)
    assert set(c) == {"GEMM1", "GEMM2"}
    assert c["GEMM1"]["units"] == 2 and c["GEMM2"]["units"] == 3
    for g in ("GEMM1", "GEMM2"):
        assert c[g]["enter"] == 100 and c[g]["decode"] == 50 and c[g]["prefetch"] == 80
        assert c[g]["to_wait"] == 40 and c[g]["mma_decode"] == 300 and c[g]["mma_to_wait"] == 60
        assert c[g]["first_period"] == 700 + 900
        assert c[g]["period"] == 700


def test_stage_summary_reads_the_same_stamps():
    st = _synthetic_fused_stages(n1=4, n2=4, kt1=6, kt2=6, bubble=0)
    lines = trace.summarize_fused_stages(st, 4 * 6)
    assert len(lines) == 2
    # every stage: the producer issued 3000 cycles before the MMA warp saw it full, and the MMA
    # warp issued 200 cycles after seeing it
    assert "load latency issue->full 3000" in lines[0] and "issue 200" in lines[0]
    assert "stage period 700 (mean 700)" in lines[1]
