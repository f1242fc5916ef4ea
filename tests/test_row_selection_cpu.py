"""The GPU tests' choice of rows to check on full-size steps, on the CPU:
the first and last pick of every token tile of every expert."""
import numpy as np

from gpu_util import tile_edge_slots


def test_tile_edges_of_a_hand_example():
    # k = 2; expert 3 holds slots 0, 2, 5, 6, 9, expert 1 slots 1, 4,
    # expert 0 slots 3, 8 and expert 2 slot 7
    ids = np.array([[3, 1], [3, 0], [1, 3], [3, 2], [0, 3]])
    # tiles of 2: expert 3 {0, 2} {5, 6} {9}, expert 1 {1, 4}, expert 0 {3, 8}, expert 2 {7}
    assert tile_edge_slots(ids, [2]).tolist() == [0, 1, 2, 3, 4, 5, 6, 7, 8, 9]
    # tiles of 8: one per expert
    assert tile_edge_slots(ids, [8]).tolist() == [0, 1, 3, 4, 7, 8, 9]
    # tiles of 3: expert 3 {0, 2, 5} {6, 9}
    assert tile_edge_slots(ids, [3]).tolist() == [0, 1, 3, 4, 5, 6, 7, 8, 9]


def test_every_tile_of_every_expert_is_represented():
    rng = np.random.default_rng(5)
    T, k, E = 700, 6, 50
    ids = np.stack([rng.choice(E, size=k, replace=False) for _ in range(T)])
    flat = ids.reshape(-1)
    for widths in ([144], [144, 160], [32]):
        sel = set(tile_edge_slots(ids, widths).tolist())
        for e in range(E):
            picks = np.flatnonzero(flat == e)          # slot order
            for W in widths:
                for t0 in range(0, picks.size, W):
                    tile = picks[t0:t0 + W]
                    assert tile[0] in sel and tile[-1] in sel
        # nothing beyond the tile ends
        ends = {int(p[t0]) for e in range(E) for p in [np.flatnonzero(flat == e)] for W in widths
                for t0 in range(0, p.size, W)}
        ends |= {int(p[min(t0 + W, p.size) - 1]) for e in range(E) for p in [np.flatnonzero(flat == e)]
                 for W in widths for t0 in range(0, p.size, W)}
        assert sel == ends
