"""Token-boundary shards of a batch over ranks, by brute force.

TEST INFRASTRUCTURE (see the package docstring). Integer arithmetic only.

[W] "Fix two: RMSNorm was never insignificant": the all-reduce that follows a
row-parallel projection is taken apart into a reduce-scatter and an
all-gather, split at token boundaries, so that each rank holds whole token
rows of the reduced tensor and normalises only those. The pages do not say
how rows are dealt out; the reading here is contiguous shards of
ceil(T / world) rows in rank order, the last non-empty one shorter (the same
shards as the 8 x 128-token configuration of the Llama-3.3-70B workload).

The oracle states that reading row by row: row t belongs to rank
t // ceil(T / world). A rank's shard is the set of rows it owns.
"""


def owner(t, T, world):
    """The rank that owns row t of a T-row batch over `world` ranks."""
    s = -(-T // world)
    return t // s


def shard_rows(T, world, rank):
    """(row0, rows) of `rank`'s shard: the rows it owns, found by testing every
    row of the batch. An empty shard starts at T."""
    mine = [t for t in range(T) if owner(t, T, world) == rank]
    if not mine:
        return T, 0
    return mine[0], len(mine)
