"""The step-kernel phase table (step_trace) on hand-made timestamps: work is
last CTA end - first CTA start, the barrier is the gap to the first CTA of the
next phase, and the last phase of the last block has no barrier."""
import io
import warnings

import numpy as np

from latency_transformer_block_gb300 import step_trace as st


def _trace(blocks=2, ctas=4):
    """Phase p of block l: CTA i starts at base + 10 i ns and ends 1000 ns + 20 i
    ns later; consecutive phases are 500 ns apart after the last end."""
    tr = np.zeros((blocks, ctas, 64), dtype=np.int64)
    t = 10_000
    expect_work, expect_bar = [], []
    for l in range(blocks):
        for _, s0, e in st.PHASES:
            starts = t + 10 * np.arange(ctas)
            ends = starts + 1000 + 20 * np.arange(ctas)
            tr[l, :, s0] = starts
            tr[l, :, e] = ends
            expect_work.append((ends.max() - starts.min()) / 1e3)
            t = int(ends.max()) + 500
            expect_bar.append(0.5)
    return tr, np.array(expect_work).reshape(blocks, -1), np.array(expect_bar).reshape(blocks, -1)


def test_phase_table_work_and_barriers():
    tr, ew, eb = _trace()
    work, bar, _ = st.phase_table(tr)
    np.testing.assert_allclose(work, ew)
    np.testing.assert_allclose(bar[:, :-1], eb[:, :-1])
    np.testing.assert_allclose(bar[0, -1], 0.5)          # down of block 0 -> QKV of block 1
    assert np.isnan(bar[-1, -1])                         # nothing follows the last block


def test_report_runs_without_warnings():
    tr, _, _ = _trace(blocks=1)
    out = io.StringIO()
    with warnings.catch_warnings():
        warnings.simplefilter("error")
        st.report(tr, out)
    text = out.getvalue()
    assert "| total |" in text and "us per block" in text
