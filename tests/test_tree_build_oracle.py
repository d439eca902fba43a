"""Pins of the tree-build oracle (no GPU)."""
import numpy as np

from oracle import tree_build as tb


def test_hand_tree():
    #        0
    #      /   \
    #     1     2
    #    / \     \
    #   3   4     5
    o = tb.build([-1, 0, 0, 1, 1, 2], seq_len=100, request=2)
    assert o["status"] == 0
    assert o["positions"] == [100, 101, 101, 102, 102, 102]
    assert o["first_child"] == [1, 3, 5, -1, -1, -1]
    assert o["next_sibling"] == [-1, 2, -1, 4, -1, -1]
    assert o["retrieve_index"] == [12, 13, 14, 15, 16, 17]
    rows = {i: [j for j in range(6) if o["mask"][i][j]] for i in range(6)}
    assert rows == {0: [0], 1: [0, 1], 2: [0, 2], 3: [0, 1, 3], 4: [0, 1, 4], 5: [0, 2, 5]}


def test_chain_is_the_topk_one_case():
    """A chain (topk = 1): causal mask, consecutive positions, next token = i + 1, no siblings."""
    N = 7
    o = tb.build([-1] + list(range(N - 1)), seq_len=5)
    assert o["positions"] == list(range(5, 5 + N))
    assert np.array_equal(np.array(o["mask"]), np.tril(np.ones((N, N), int)))
    assert o["first_child"] == list(range(1, N)) + [-1]
    assert o["next_sibling"] == [-1] * N


def test_links_reproduce_the_parent_array():
    rng = np.random.default_rng(4)
    for _ in range(100):
        N = int(rng.integers(1, 40))
        par = [-1] + [int(rng.integers(0, i)) for i in range(1, N)]
        o = tb.build(par, seq_len=0)
        for i in range(N):
            kids, c = [], o["first_child"][i]
            while c != -1:
                kids.append(c)
                c = o["next_sibling"][c]
            assert kids == [j for j in range(N) if par[j] == i]
            # mask row = the ancestor chain; its size is depth + 1
            assert sum(o["mask"][i]) == o["positions"][i] + 1


def test_invalid_trees():
    for par in ([0, 0], [-1, 1], [-1, 0, 5], [-1, -1], []):
        o = tb.build(par, seq_len=3)
        assert o["status"] == tb.BAD_TREE
        assert o["first_child"] == [-1] * len(par) and o["next_sibling"] == [-1] * len(par)
