"""Host side of the timeline tracing tool: interval arithmetic on synthetic stamps (CPU)."""

import numpy as np

from chunked_prefill_causal_gb300 import timeline


def test_intervals_from_synthetic_stamps():
    # period 1000 cycles per tile; softmax S->ld 10, exps 500, store 20; issuer sees P 30 later,
    # turn 40 later, P V issue 200, Q K^T issue 300, S ready 5 cycles after the block is issued
    buf = np.zeros((4, 64, 4), dtype=np.int64)
    for x in range(2):
        for j in range(64):
            s0 = 1000 * j + 500 * x
            buf[2 + x, j] = [s0, s0 + 10, s0 + 510, s0 + 530]
            seen = 1000 * (j - 1) + 500 * x + 530 + 30
            buf[x, j, 0] = seen
            buf[x, j, 1] = seen + 40
            buf[x, j, 3] = seen + 240
            buf[x, j, 2] = s0 - 5
    iv = timeline.intervals(buf)
    for t in "AB":
        assert iv[f"{t}.softmax: S ready -> S in registers"] == 10
        assert iv[f"{t}.softmax: exponentials"] == 500
        assert iv[f"{t}.softmax: store P + signal"] == 20
        assert iv[f"{t}.issuer: P signalled -> seen"] == 30
        assert iv[f"{t}.issuer: seen -> turn"] == 40
        assert iv[f"{t}.issuer: turn -> P V issued (8 TS MMAs)"] == 200
        assert iv[f"{t}.issuer: block issued -> S ready"] == 5
        assert iv[f"{t}.period (S ready to S ready)"] == 1000
