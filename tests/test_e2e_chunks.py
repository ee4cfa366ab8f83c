"""Host logic of the end-to-end step (bench.py): its copy chunks cover every layer's inputs and outputs once.

Layer 0's inputs go up before the plan and the rest in the upload chunks; outputs go down in the download chunks
and, from the last cut on, after the step.  A layer copied twice would double-count bytes; one never copied would
leave its inputs or outputs stale."""
import pytest

import bench


@pytest.mark.parametrize("L", list(range(1, 70)))
def test_chunks_partition_the_layers(L):
    ups, cuts = bench.e2e_chunks(L)
    # uploads: layer 0 alone, then [ups[c], ups[c + 1]) and the last chunk up to L
    up_layers = [0]
    for c, lo in enumerate(ups):
        hi = ups[c + 1] if c + 1 < len(ups) else L
        assert lo < hi
        up_layers += list(range(lo, hi))
    assert up_layers == list(range(L))
    if ups:
        assert ups[0] == 1 and all(b == 2 * a for a, b in zip(ups, ups[1:]))
    # downloads: [cuts[c - 1], cuts[c]) before layer cuts[c] runs, then the tail after the step
    down_layers = []
    for c, hi in enumerate(cuts):
        lo = cuts[c - 1] if c else 0
        assert lo < hi
        down_layers += list(range(lo, hi))
    down_layers += list(range(cuts[-1] if cuts else 0, L))
    assert down_layers == list(range(L))
    # the exposed copies at each end are one layer's
    assert not cuts or L - cuts[-1] == 1


def test_chunks_of_the_28_layer_step():
    assert bench.e2e_chunks(28) == ([1, 2, 4, 8, 16], [12, 20, 24, 26, 27])
