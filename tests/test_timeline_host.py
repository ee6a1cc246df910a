"""Host side of the %globaltimer timeline tool: its analysis of the stamp
records, on a hand-made record of two kv-head lanes and four launches."""
import numpy as np

from paged_decode_attention_cache_gb300 import timeline as T


def _record(n_launches=4, grid=4):
    rec = np.zeros((T.LAUNCHES, T.CTAS, T.WORDS), dtype=np.int64)
    for l in range(n_launches):
        t0 = 10_000 + l * 20_000          # launch l starts at t0 (ns)
        for c in range(grid):
            r = rec[l, c]
            r[0], r[1], r[2], r[3] = t0, t0 + 500, t0 + 1_000, t0 + 2_000
            nseg = 2 if c == 1 else 1
            for k in range(nseg):
                base = 4 + 4 * k
                r[base:base + 4] = [t0 + 2_000 + 5_000 * k, t0 + 6_000 + 5_000 * k, t0 + 6_500 + 5_000 * k,
                                    t0 + 7_000 + 5_000 * k + 100 * c]
            combined_last = 1 if c == 2 else 0
            r[28] = nseg | (combined_last << (8 + nseg - 1)) | (1 << 16)
            r[29] = 40 | (20 << 16) if nseg == 2 else 60
    return rec


def test_phases_are_relative_to_the_previous_launchs_last_cta():
    grid, R, periods, nseg, blocks, comb_end, tails = T.analyse(_record(), 4, hkv=2)
    assert grid == 4
    # launches 2 and 3 are reported; the last CTA (1: two segments) ends at t0 + 12_100
    assert R.shape == (2, 4, 6)
    assert np.allclose(periods, 20.0)
    prev_end_to_entry = (10_000 + 2 * 20_000) - (10_000 + 1 * 20_000 + 12_100)
    assert np.isclose(R[0, 0, 0], prev_end_to_entry / 1e3)
    # the end column of CTA 1 is its second segment's end
    assert np.isclose(R[0, 1, 5], (12_100 - 12_100 + 20_000) / 1e3)
    assert (nseg[:, 1] == 2).all() and (nseg[:, 0] == 1).all()
    assert (blocks[:, 1] == 60).all() and (blocks[:, 0] == 60).all()
    assert comb_end[:, 2].all() and not comb_end[:, 0].any()
    # the piece bit is set for segment 0 only: CTA 1's last (second) segment is a whole pair;
    # merged at 6_000 + 5_000 k, published 500 later, end 1_000 + 100 c after the merge
    assert tails["piece"][:, [0, 2, 3]].all() and not tails["piece"][:, 1].any()
    assert np.allclose(tails["merged_to_published"][:, [0, 2, 3]], 0.5)
    assert np.isnan(tails["merged_to_published"][:, 1]).all()
    assert np.allclose(tails["published_to_end"][:, 3], 0.8)
    assert np.allclose(tails["merged_to_end"][:, 1], 1.1)


def test_report_lists_every_lane_range():
    rec = _record()
    grid, R, periods, nseg, blocks, comb_end, tails = T.analyse(rec, 4, hkv=2)

    class B:
        schedule = "balanced"

    text = T.report("w", B(), grid, R, periods, nseg, blocks, comb_end, 2, 0, tails)
    rows = [l for l in text.splitlines() if l.startswith("| 0 |") or l.startswith("| 1 |")]
    assert len(rows) == 2
    assert "Launch period" in text
    assert "piece that combines its pair" in text
