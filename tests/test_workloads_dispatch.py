"""Host logic of the quantize-once dispatch inputs: the routed-row -> token index."""
import numpy as np

import workloads


def test_dispatch_index_is_the_routing():
    T = 3000
    choices = workloads.route_choices(T)
    counts = workloads.route_counts(T)
    assert np.array_equal(np.bincount(choices.reshape(-1), minlength=workloads.EXPERTS), counts)
    assert all(len(set(r)) == workloads.TOPK for r in choices[:200])          # distinct experts
    offs = workloads.padded_offsets(counts, 32)
    idx = workloads.dispatch_index(choices, offs)
    assert idx.size == offs[-1]
    assert np.array_equal(np.bincount(idx[idx >= 0], minlength=T), np.full(T, workloads.TOPK))
    for e in range(workloads.EXPERTS):
        seg = idx[offs[e]:offs[e + 1]]
        real, pad = seg[:counts[e]], seg[counts[e]:]
        assert (pad == -1).all() and (real >= 0).all()
        assert (np.diff(real) > 0).all()                                      # token order within an expert
        assert all(e in choices[t] for t in real[:20])


def test_route_counts_unchanged_by_the_refactor():
    # the 16384-token Zipf(1.1) routing the MoE configuration is quoted on
    c = workloads.route_counts(16384)
    assert c.sum() == 131072 and c.min() == 173 and c.max() == 14749


def test_dispatch_dest_inverts_dispatch_index():
    T = 3000
    choices = workloads.route_choices(T)
    counts = np.bincount(choices.reshape(-1), minlength=workloads.EXPERTS)
    for align in (1, 32):
        offs = workloads.padded_offsets(counts, align)
        idx = workloads.dispatch_index(choices, offs)
        dest = workloads.dispatch_dest(choices, offs)
        assert dest.shape == choices.shape and dest.dtype == np.int32
        # every (token, k) names a distinct real routed row of its own token and expert
        assert len(np.unique(dest)) == dest.size
        assert np.array_equal(idx[dest], np.repeat(np.arange(T)[:, None], workloads.TOPK, axis=1))
        e_of_row = np.searchsorted(offs, dest, side="right") - 1
        assert np.array_equal(e_of_row, choices)
