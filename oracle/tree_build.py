"""Tree-verify inputs from parent lists, restated in plain Python.

Test infrastructure only: imported by tests/, by the package smoke check and
by the benchmark's CPU-baseline leg.  The product path never imports it.

Source: "从 EAGLE 到 DFlash 2：SGLang 与 SpecForge 的投机解码训练和推理",
section 2.4 (a flattened tree: every node sees only the committed history, its
ancestors and itself; position ids follow the path depth, not the array
index) and section 3.4 (tree construction produces the mask, the positions
and the retrieve index / next-token / next-sibling arrays that drive the
verify walk).  Siblings are taken in node-index order, the order in which the
tree walk of the verify step visits them.
"""
from __future__ import annotations

from typing import Sequence

BAD_TREE = 4  # SV_DEV_BAD_TREE


def valid(parents: Sequence[int]) -> bool:
    """Node 0 is the root (parent -1); every other node's parent comes before it."""
    if len(parents) == 0 or parents[0] != -1:
        return False
    return all(0 <= parents[i] < i for i in range(1, len(parents)))


def build(parents: Sequence[int], seq_len: int, request: int = 0) -> dict:
    """Outputs for one request of N nodes.

    depth[i] = 0 for the root, depth[parent] + 1 otherwise; positions[i] =
    seq_len + depth[i]; mask[i][j] = 1 iff j is i or one of its ancestors;
    retrieve_index[i] = request * N + i; first_child[i] = the lowest-index
    child of i (-1 if none); next_sibling[i] = the lowest-index node after i
    with the same parent (-1 if none).  An invalid tree gives status
    BAD_TREE, positions seq_len, an identity mask and -1 links.
    """
    N = len(parents)
    out = {"positions": [seq_len] * N, "mask": [[1 if i == j else 0 for j in range(N)] for i in range(N)],
           "retrieve_index": [request * N + i for i in range(N)], "first_child": [-1] * N,
           "next_sibling": [-1] * N, "status": 0}
    if not valid(parents):
        out["status"] = BAD_TREE
        return out
    depth = [0] * N
    for i in range(1, N):
        depth[i] = depth[parents[i]] + 1
    out["positions"] = [seq_len + d for d in depth]
    for i in range(N):
        j = i
        while j != -1:
            out["mask"][i][j] = 1
            j = parents[j]
    for i in range(1, N):
        p = parents[i]
        if out["first_child"][p] == -1:
            out["first_child"][p] = i
        later = [j for j in range(i + 1, N) if parents[j] == p]
        out["next_sibling"][i] = later[0] if later else -1
    return out
